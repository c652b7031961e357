/*
 * dsa_oracle.h -- entry points of the CPU oracle (test infrastructure only;
 * see dsa_oracle.c for the definition each one follows). Return 0 on
 * success, -1 on an invalid argument, -2 when host memory runs out.
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int dsa_oracle_block_scores(const float *logits, int64_t rows, int64_t width,
                            int64_t ld_logits, const int32_t *row_ks,
                            const int32_t *row_ke, int32_t block_size,
                            int32_t row_repeat, int32_t pin_newest,
                            float *scores, int64_t ld_scores);

int dsa_oracle_select(const float *logits, int64_t rows, int64_t width,
                      int64_t ld_logits, const int32_t *row_ks,
                      const int32_t *row_ke, int32_t topk_blocks,
                      int32_t block_size, int32_t row_repeat,
                      int32_t pin_newest, int32_t *out, int64_t ld_out,
                      float *scores, int64_t ld_scores);

int dsa_oracle_select_sharded(const float *logits, int32_t shards,
                              int64_t rows, int64_t local_width,
                              int64_t ld_logits, int64_t shard_stride,
                              const int32_t *global_row_ke,
                              int32_t global_block_size,
                              int32_t max_global_blocks, int32_t row_repeat,
                              int32_t topk_blocks, int32_t *out,
                              int64_t ld_out, float *scores, int64_t ld_scores);

int dsa_oracle_mask(float *logits, int64_t rows, int64_t width, int64_t ld_logits,
                    const int32_t *row_ks, const int32_t *row_ke,
                    const int32_t *cand, int64_t topk, int64_t ld_cand,
                    int32_t block_size, int32_t row_repeat);

int dsa_oracle_mask_sharded(float *logits, int32_t shards, int64_t rows, int64_t local_width,
                            int64_t ld_logits, int64_t shard_stride,
                            const int32_t *global_row_ke, int32_t global_block_size,
                            int32_t row_repeat, const int32_t *cand, int64_t topk,
                            int64_t ld_cand);

/* The DCP form with global starts (reading R12 in dsa_oracle.c); a NULL
 * global_row_ks is the same as the functions above. */
int dsa_oracle_select_sharded_starts(const float *logits, int32_t shards, int64_t rows,
                                     int64_t local_width, int64_t ld_logits,
                                     int64_t shard_stride, const int32_t *global_row_ks,
                                     const int32_t *global_row_ke, int32_t global_block_size,
                                     int32_t max_global_blocks, int32_t row_repeat,
                                     int32_t topk_blocks, int32_t *out, int64_t ld_out,
                                     float *scores, int64_t ld_scores);

int dsa_oracle_mask_sharded_starts(float *logits, int32_t shards, int64_t rows,
                                   int64_t local_width, int64_t ld_logits,
                                   int64_t shard_stride, const int32_t *global_row_ks,
                                   const int32_t *global_row_ke, int32_t global_block_size,
                                   int32_t row_repeat, const int32_t *cand, int64_t topk,
                                   int64_t ld_cand);

/* bf16 logits (dsa_oracle_bf16.c): the same definitions on the exact fp32
 * widening of the bf16 values; scores are bf16 bit patterns. */
int dsa_oracle_block_scores_bf16(const uint16_t *logits, int64_t rows, int64_t width,
                                 int64_t ld_logits, const int32_t *row_ks,
                                 const int32_t *row_ke, int32_t block_size,
                                 int32_t row_repeat, int32_t pin_newest, uint16_t *scores,
                                 int64_t ld_scores);

int dsa_oracle_select_bf16(const uint16_t *logits, int64_t rows, int64_t width,
                           int64_t ld_logits, const int32_t *row_ks, const int32_t *row_ke,
                           int32_t topk_blocks, int32_t block_size, int32_t row_repeat,
                           int32_t pin_newest, int32_t *out, int64_t ld_out, uint16_t *scores,
                           int64_t ld_scores);

int dsa_oracle_select_sharded_bf16(const uint16_t *logits, int32_t shards, int64_t rows,
                                   int64_t local_width, int64_t ld_logits,
                                   int64_t shard_stride, const int32_t *global_row_ke,
                                   int32_t global_block_size, int32_t max_global_blocks,
                                   int32_t row_repeat, int32_t topk_blocks, int32_t *out,
                                   int64_t ld_out, uint16_t *scores, int64_t ld_scores);

int dsa_oracle_mask_bf16(uint16_t *logits, int64_t rows, int64_t width, int64_t ld_logits,
                         const int32_t *row_ks, const int32_t *row_ke, const int32_t *cand,
                         int64_t topk, int64_t ld_cand, int32_t block_size, int32_t row_repeat);

int dsa_oracle_mask_sharded_bf16(uint16_t *logits, int32_t shards, int64_t rows,
                                 int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                                 const int32_t *global_row_ke, int32_t global_block_size,
                                 int32_t row_repeat, const int32_t *cand, int64_t topk,
                                 int64_t ld_cand);

#ifdef __cplusplus
}
#endif

#endif /* DSA_ORACLE_H */
