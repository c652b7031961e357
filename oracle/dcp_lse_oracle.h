/*
 * dcp_lse_oracle.h -- entry points of the CPU oracle for the DCP LSE
 * correction (test infrastructure only; dcp_lse_oracle.c states the
 * definition). Layouts are dense: out [B, H, Dh], outs [N, B, H, Dh],
 * lses [N, B, H], new_out / merged [H, B, Dh] (head-major), lse_out [B, H].
 * Return 0 on success, -1 on an invalid argument.
 */
#ifndef DCP_LSE_ORACLE_H
#define DCP_LSE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int dcp_oracle_correct_attn_out(const float *out, const float *lses, int32_t shards,
                                int64_t batch, int64_t heads, int64_t head_dim,
                                int32_t rank, double *new_out, double *lse_out);

int dcp_oracle_merge_attn_out(const float *outs, const float *lses, int32_t shards,
                              int64_t batch, int64_t heads, int64_t head_dim,
                              double *merged, double *lse_out);

#ifdef __cplusplus
}
#endif

#endif /* DCP_LSE_ORACLE_H */
