/*
 * dsa_dcp_attn.h -- C ABI of the DCP partial-attention LSE correction in the
 * GB300 (sm_103a) library libdsa_cb.so (status codes and the conventions on
 * device pointers and streams are those of dsa_cb.h).
 *
 * The operation (page "sgl-project--sglang/python/sglang/srt/layers/dcp/
 * kernels.py": _correct_attn_cp_out_kernel and correct_attn_out). Under
 * decode context parallelism each of N shards runs attention over its own
 * share of the keys and gets a partial output o_n[b,h,:] and a base-2
 * log-sum-exp l_n[b,h]. For every token b and head h:
 *   x_n = l_n, with NaN and +inf read as -inf;
 *   m   = max_n x_n, or 0 when every x_n is -inf;
 *   F   = log2(sum_n 2^(x_n - m)) + m            (combined LSE);
 *   f_n = 2^(l_n - F), with a NaN or +inf exponent read as -inf, so that
 *         the share is 0.
 * dsa_correct_attn_out writes F and f_i * o_i for one shard i (the page's
 * kernel); dsa_merge_attn_out writes sum_n f_n * o_n, the cross-shard sum
 * that the page leaves to a collective, for all N shards held on one GPU as
 * a leading axis. A token with no finite LSE gets F = -inf and an output of
 * f * o = 0 * o.
 *
 * Arithmetic is fp32 (exp2f / log2f, fused multiply-adds for the merge in
 * shard order); bf16 outputs are widened on load and rounded to nearest even
 * on store. Results therefore match an exact evaluation within fp32 (or
 * bf16) rounding, not bit for bit.
 *
 * Layouts: every tensor is addressed through element strides, so views
 * (e.g. a [B, 1, H, D] output squeezed to [B, H, D], or a transposed LSE
 * buffer) are passed without copies. The output is written head-major as on
 * the page: element (h, b, d) at new_out + h * new_sh + b * new_sb + d * new_sd.
 * With unit stride in the head dimension, 16-byte aligned rows and a head
 * dimension that is a whole number of 16-byte vectors, data moves in 16-byte
 * vectors; any other layout is still accepted and moves element by element.
 */
#ifndef DSA_DCP_ATTN_H
#define DSA_DCP_ATTN_H

#include <stdint.h>

#include "dsa_cb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the attention outputs (the LSEs are always fp32). */
typedef enum {
    DSA_DTYPE_F32 = 0,
    DSA_DTYPE_BF16 = 1
} dsa_dtype;

/* Largest shard count N the two entry points accept (one lane of a warp per
 * shard); larger N returns DSA_EUNSUPPORTED. */
int32_t dsa_attn_max_shards(void);

/*
 * dsa_correct_attn_out -- the correction of one shard's partial output.
 *
 *   out       [batch, heads, head_dim] of `dtype`: shard `rank`'s partial
 *             output; element (b, h, d) at out + b*out_sb + h*out_sh + d*out_sd.
 *   lses      [shards, batch, heads] fp32 base-2 LSEs of all shards;
 *             element (n, b, h) at lses + n*lse_sn + b*lse_sb + h*lse_sh.
 *   rank      0 <= rank < shards: the shard `out` belongs to.
 *   new_out   [heads, batch, head_dim] of `dtype`: f_rank * out, written at
 *             new_out + h*new_sh + b*new_sb + d*new_sd. Must not overlap
 *             out (or lses / lse_out).
 *   lse_out   [batch, heads] fp32 combined LSE F at lse_out + b*lo_sb +
 *             h*lo_sh, or NULL to skip it.
 *
 * batch == 0 or heads == 0: DSA_OK, nothing written. head_dim == 0: only
 * lse_out is written (out and new_out may then be NULL). DSA_EINVAL for an
 * unknown dtype, shards < 1, rank outside [0, shards), negative sizes, or a
 * NULL lses (or NULL out / new_out when head_dim > 0). DSA_EUNSUPPORTED for
 * shards > dsa_attn_max_shards() or head_dim >= 2^31.
 */
dsa_status dsa_correct_attn_out(const void *out, int32_t dtype, int64_t batch,
                                int64_t heads, int64_t head_dim, int64_t out_sb,
                                int64_t out_sh, int64_t out_sd, const float *lses,
                                int32_t shards, int64_t lse_sn, int64_t lse_sb,
                                int64_t lse_sh, int32_t rank, void *new_out,
                                int64_t new_sh, int64_t new_sb, int64_t new_sd,
                                float *lse_out, int64_t lo_sb, int64_t lo_sh,
                                void *stream);

/*
 * dsa_merge_attn_out -- the corrected partial outputs of all shards, summed.
 *
 *   outs      [shards, batch, heads, head_dim] of `dtype`; element (n, b, h, d)
 *             at outs + n*outs_sn + b*outs_sb + h*outs_sh + d*outs_sd.
 *   lses      as for dsa_correct_attn_out.
 *   merged    [heads, batch, head_dim] of `dtype`: sum_n f_n * o_n (fp32
 *             fused multiply-adds in shard order, then one rounding to
 *             `dtype`), at merged + h*m_sh + b*m_sb + d*m_sd. Must not
 *             overlap outs.
 *   lse_out   as for dsa_correct_attn_out.
 *
 * Sizes, NULL rules and errors as for dsa_correct_attn_out (without rank).
 */
dsa_status dsa_merge_attn_out(const void *outs, int32_t dtype, int32_t shards,
                              int64_t batch, int64_t heads, int64_t head_dim,
                              int64_t outs_sn, int64_t outs_sb, int64_t outs_sh,
                              int64_t outs_sd, const float *lses, int64_t lse_sn,
                              int64_t lse_sb, int64_t lse_sh, void *merged,
                              int64_t m_sh, int64_t m_sb, int64_t m_sd,
                              float *lse_out, int64_t lo_sb, int64_t lo_sh,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_DCP_ATTN_H */
