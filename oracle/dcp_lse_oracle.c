/*
 * dcp_lse_oracle.c -- plain, single-threaded CPU oracle for the DCP
 * partial-attention LSE correction.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. No product code path
 * calls it, and it shares no code, header, table or helper with the CUDA
 * implementation.
 *
 * Source (web page):
 *   [SG]  "sgl-project--sglang/python/sglang/srt/layers/dcp/kernels.py" --
 *         _correct_attn_cp_out_kernel and correct_attn_out (the partial-
 *         attention LSE correction of the MLA decode-context-parallel path).
 *
 * What it computes, for every (b, h), from the base-2 log-sum-exps lses[n,b,h]
 * of the N context shards and the partial output out[b,h,:] of shard i:
 *   1. x_n = lses[n,b,h], with NaN and +inf read as -inf;
 *   2. m = max_n x_n, or 0 when every x_n is -inf;
 *   3. F = log2(sum_n 2^(x_n - m)) + m        (the combined LSE);
 *   4. d = lses[i,b,h] - F, the raw local value, with a NaN or +inf
 *      difference read as -inf;
 *   5. f = 2^d                                  (shard i's share);
 *   6. lse_out[b,h] = F and new_out[h,b,:] = f * out[b,h,:] (the output is
 *      written head-major, [H, B, Dh], as on the page).
 * Readings where the page is silent (each listed in the design notes):
 *   L1 the arithmetic is exact here (double precision, libm exp2/log2); the
 *      page computes in fp32, so the CUDA path is compared within a
 *      tolerance derived from fp32 rounding.
 *   L2 the "cross-rank reduction" that follows the correction is a sum:
 *      merged[h,b,:] = sum_n f_n * out_n[b,h,:], f_n being step 5 for shard
 *      n. (The shares f_n add up to 1 whenever some x_n is finite, so the
 *      sum is the attention output over all shards' keys.)
 *   L3 N is any positive count (the page rounds it to a power of two only
 *      to size a vector).
 */
#include "dcp_lse_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* Step 1: NaN and +inf count as -inf. */
static double sanitize(double x)
{
    if (isnan(x) || x == INFINITY)
        return -INFINITY;
    return x;
}

/* Steps 1-3 for one (b, h): the combined LSE of lse[0..n) (stride step). */
static double combined_lse(const float *lse, int64_t step, int32_t n)
{
    double m = -INFINITY, acc = 0.0;
    int32_t k;
    for (k = 0; k < n; ++k) {
        double x = sanitize((double)lse[k * step]);
        if (x > m)
            m = x;
    }
    if (m == -INFINITY)
        m = 0.0;
    for (k = 0; k < n; ++k)
        acc += exp2(sanitize((double)lse[k * step]) - m);
    return log2(acc) + m;
}

/* Steps 4-5: the share of the shard whose LSE is local. */
static double share(double local, double final_lse)
{
    double d = local - final_lse;
    if (isnan(d) || d == INFINITY)
        d = -INFINITY;
    return exp2(d);
}

int dcp_oracle_correct_attn_out(const float *out, const float *lses, int32_t shards,
                                int64_t batch, int64_t heads, int64_t head_dim,
                                int32_t rank, double *new_out, double *lse_out)
{
    int64_t b, h, c;
    if (shards < 1 || rank < 0 || rank >= shards || batch < 0 || heads < 0 || head_dim < 0)
        return -1;
    for (b = 0; b < batch; ++b)
        for (h = 0; h < heads; ++h) {
            const float *col = lses + b * heads + h;   /* lses[., b, h] */
            int64_t step = batch * heads;
            double F = combined_lse(col, step, shards);
            double f = share((double)col[rank * step], F);
            const float *src = out + (b * heads + h) * head_dim;
            double *dst = new_out + (h * batch + b) * head_dim;
            lse_out[b * heads + h] = F;
            for (c = 0; c < head_dim; ++c)
                dst[c] = f * (double)src[c];
        }
    return 0;
}

int dcp_oracle_merge_attn_out(const float *outs, const float *lses, int32_t shards,
                              int64_t batch, int64_t heads, int64_t head_dim,
                              double *merged, double *lse_out)
{
    int64_t b, h, c;
    int32_t n;
    if (shards < 1 || batch < 0 || heads < 0 || head_dim < 0)
        return -1;
    for (b = 0; b < batch; ++b)
        for (h = 0; h < heads; ++h) {
            const float *col = lses + b * heads + h;
            int64_t step = batch * heads;
            double F = combined_lse(col, step, shards);
            double *dst = merged + (h * batch + b) * head_dim;
            lse_out[b * heads + h] = F;
            for (c = 0; c < head_dim; ++c)
                dst[c] = 0.0;
            /* L2: the cross-shard reduction is the sum of the corrected
             * partial outputs. */
            for (n = 0; n < shards; ++n) {
                double f = share((double)col[n * step], F);
                const float *src = outs + ((n * batch + b) * heads + h) * head_dim;
                for (c = 0; c < head_dim; ++c)
                    dst[c] += f * (double)src[c];
            }
        }
    return 0;
}
