/*
 * dsa_oracle_bf16.c -- the CPU oracle's entry points for bf16 logits.
 *
 * TEST INFRASTRUCTURE, like dsa_oracle.c (only the tests, the package smoke
 * check and the benchmark's CPU-baseline leg load it; no product code path
 * calls it; it shares nothing with the CUDA implementation).
 *
 * Source: the page "launcher/dcp2/diffs/02-model_executor_kernels_attention_
 * dsa_candidate_blocks.py.diff" -- _block_scores allocates the scores with
 * the logits' own dtype (logits.new_empty), so bf16 logits give bf16 scores;
 * everything else is the fp32 definition of dsa_oracle.c.
 *
 * Readings (listed in the design notes with the others):
 *   R9  a bf16 logit is the real number whose fp32 encoding has the bf16
 *       bits as its upper 16 bits (the exact widening); selection runs on
 *       those values, so it is the fp32 definition applied to them.
 *   R10 a bf16 score is the upper half of the fp32 score: exact, because a
 *       block max is one of the block's values (or +-inf); a NaN score is
 *       the canonical bf16 quiet NaN 0x7FC0.
 *   R11 masking writes bf16 -inf (0xFF80) and leaves kept logits untouched.
 */
#include "dsa_oracle.h"

#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float bf16_value(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

static uint16_t bf16_bits(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

/* The [n_outer, n_inner] block of bf16 values at src (outer stride ld) as
 * dense fp32. */
static float *widen(const uint16_t *src, int64_t n_outer, int64_t n_inner, int64_t ld)
{
    int64_t i, j;
    float *dst = (float *)malloc((size_t)(n_outer * n_inner > 0 ? n_outer * n_inner : 1) *
                                 sizeof(float));
    if (!dst)
        return NULL;
    for (i = 0; i < n_outer; ++i)
        for (j = 0; j < n_inner; ++j)
            dst[i * n_inner + j] = bf16_value(src[i * ld + j]);
    return dst;
}

/* fp32 scores [rows, nb] (dense) into bf16 scores with row stride ld. */
static void narrow(const float *src, int64_t rows, int64_t nb, uint16_t *dst, int64_t ld)
{
    int64_t i, j;
    for (i = 0; i < rows; ++i)
        for (j = 0; j < nb; ++j)
            dst[i * ld + j] = bf16_bits(src[i * nb + j]);
}

static int64_t nblocks(int64_t width, int32_t bs) { return bs > 0 ? (width + bs - 1) / bs : 0; }

int dsa_oracle_block_scores_bf16(const uint16_t *logits, int64_t rows, int64_t width,
                                 int64_t ld_logits, const int32_t *row_ks,
                                 const int32_t *row_ke, int32_t block_size,
                                 int32_t row_repeat, int32_t pin_newest, uint16_t *scores,
                                 int64_t ld_scores)
{
    int64_t nb = nblocks(width, block_size);
    float *x, *s;
    int rc;
    if (rows < 0 || width < 0 || block_size < 1 || ld_logits < width)
        return -1;
    x = widen(logits, rows, width, ld_logits);
    s = (float *)malloc((size_t)(rows * nb > 0 ? rows * nb : 1) * sizeof(float));
    if (!x || !s) {
        free(x);
        free(s);
        return -2;
    }
    rc = dsa_oracle_block_scores(x, rows, width, width, row_ks, row_ke, block_size, row_repeat,
                                 pin_newest, s, nb);
    if (rc == 0)
        narrow(s, rows, nb, scores, ld_scores);
    free(x);
    free(s);
    return rc;
}

int dsa_oracle_select_bf16(const uint16_t *logits, int64_t rows, int64_t width,
                           int64_t ld_logits, const int32_t *row_ks, const int32_t *row_ke,
                           int32_t topk_blocks, int32_t block_size, int32_t row_repeat,
                           int32_t pin_newest, int32_t *out, int64_t ld_out, uint16_t *scores,
                           int64_t ld_scores)
{
    int64_t nb = nblocks(width, block_size);
    float *x, *s;
    int rc;
    if (rows < 0 || width < 0 || block_size < 1 || ld_logits < width)
        return -1;
    x = widen(logits, rows, width, ld_logits);
    s = (float *)malloc((size_t)(rows * nb > 0 ? rows * nb : 1) * sizeof(float));
    if (!x || !s) {
        free(x);
        free(s);
        return -2;
    }
    rc = dsa_oracle_select(x, rows, width, width, row_ks, row_ke, topk_blocks, block_size,
                           row_repeat, pin_newest, out, ld_out, scores ? s : NULL,
                           nb > 0 ? nb : 1);
    if (rc == 0 && scores)
        narrow(s, rows, nb, scores, ld_scores);
    free(x);
    free(s);
    return rc;
}

int dsa_oracle_select_sharded_bf16(const uint16_t *logits, int32_t shards, int64_t rows,
                                   int64_t local_width, int64_t ld_logits,
                                   int64_t shard_stride, const int32_t *global_row_ke,
                                   int32_t global_block_size, int32_t max_global_blocks,
                                   int32_t row_repeat, int32_t topk_blocks, int32_t *out,
                                   int64_t ld_out, uint16_t *scores, int64_t ld_scores)
{
    int64_t nbg = max_global_blocks > 1 ? max_global_blocks : 1;
    int64_t d;
    float *x, *s;
    int rc;
    if (shards < 1 || rows < 0 || local_width < 0 || ld_logits < local_width)
        return -1;
    x = (float *)malloc((size_t)(shards * rows * local_width > 0 ? shards * rows * local_width
                                                                   : 1) * sizeof(float));
    s = (float *)malloc((size_t)(rows * nbg > 0 ? rows * nbg : 1) * sizeof(float));
    if (!x || !s) {
        free(x);
        free(s);
        return -2;
    }
    for (d = 0; d < shards; ++d) {
        float *part = widen(logits + d * shard_stride, rows, local_width, ld_logits);
        if (!part) {
            free(x);
            free(s);
            return -2;
        }
        memcpy(x + d * rows * local_width, part, (size_t)(rows * local_width) * sizeof(float));
        free(part);
    }
    rc = dsa_oracle_select_sharded(x, shards, rows, local_width, local_width,
                                   rows * local_width, global_row_ke, global_block_size,
                                   max_global_blocks, row_repeat, topk_blocks, out, ld_out,
                                   scores ? s : NULL, nbg);
    if (rc == 0 && scores)
        narrow(s, rows, nbg, scores, ld_scores);
    free(x);
    free(s);
    return rc;
}

int dsa_oracle_mask_bf16(uint16_t *logits, int64_t rows, int64_t width, int64_t ld_logits,
                         const int32_t *row_ks, const int32_t *row_ke, const int32_t *cand,
                         int64_t topk, int64_t ld_cand, int32_t block_size, int32_t row_repeat)
{
    float *x;
    int rc;
    if (rows < 0 || width < 0 || ld_logits < width)
        return -1;
    x = widen(logits, rows, width, ld_logits);
    if (!x)
        return -2;
    rc = dsa_oracle_mask(x, rows, width, width, row_ks, row_ke, cand, topk, ld_cand,
                         block_size, row_repeat);
    if (rc == 0)
        narrow(x, rows, width, logits, ld_logits);
    free(x);
    return rc;
}

int dsa_oracle_mask_sharded_bf16(uint16_t *logits, int32_t shards, int64_t rows,
                                 int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                                 const int32_t *global_row_ke, int32_t global_block_size,
                                 int32_t row_repeat, const int32_t *cand, int64_t topk,
                                 int64_t ld_cand)
{
    float *x;
    int64_t d;
    int rc;
    if (shards < 1 || rows < 0 || local_width < 0 || ld_logits < local_width)
        return -1;
    x = (float *)malloc((size_t)(shards * rows * local_width > 0 ? shards * rows * local_width
                                                                   : 1) * sizeof(float));
    if (!x)
        return -2;
    for (d = 0; d < shards; ++d) {
        float *part = widen(logits + d * shard_stride, rows, local_width, ld_logits);
        if (!part) {
            free(x);
            return -2;
        }
        memcpy(x + d * rows * local_width, part, (size_t)(rows * local_width) * sizeof(float));
        free(part);
    }
    rc = dsa_oracle_mask_sharded(x, shards, rows, local_width, local_width, rows * local_width,
                                 global_row_ke, global_block_size, row_repeat, cand, topk,
                                 ld_cand);
    if (rc == 0)
        for (d = 0; d < shards; ++d)
            narrow(x + d * rows * local_width, rows, local_width, logits + d * shard_stride,
                   ld_logits);
    free(x);
    return rc;
}
