/*
 * dsa_oracle.c -- plain, single-threaded CPU oracle for DSA candidate-block
 * selection.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. No product code path
 * calls it, and it shares no code, header, table or helper with the CUDA
 * implementation.
 *
 * Sources (web pages):
 *   [CB]  "launcher/dcp2/diffs/02-model_executor_kernels_attention_dsa_
 *         candidate_blocks.py.diff" -- vLLM-fork candidate_blocks.py:
 *         _max_with_nan, _block_scores_kernel, _block_scores,
 *         _select_candidate_blocks_impl (docstring and DCP branch),
 *         _store_candidates_kernel launch.
 *   [SG]  "sgl-project--sglang/python/sglang/srt/layers/dcp/kernels.py" --
 *         create_triton_kv_indices_for_dcp_triton and
 *         update_kv_lens_and_indices (interleave-1 token placement).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *   R1 block origin is request-local: block b of a row covers columns
 *      [s + b*bs, s + (b+1)*bs) -- the pin formula (end-start-1)//BLOCK_SIZE
 *      in [CB] _block_scores_kernel names the newest block only then.
 *   R2 NaN propagates through the block max ([CB] _max_with_nan) and ranks
 *      above +inf in selection; a NaN score is written as the canonical quiet
 *      NaN 0x7FC00000.
 *   R3 bounds are clamped: e = min(ke, width), s = min(max(ks, 0), e).
 *   R4 max and ranking use one total order: -inf < ... < -0 < +0 < ... < +inf
 *      < NaN (all NaNs equal).
 *   R5 equal scores rank the lower block id first.
 *   R6 an output slot is -1 when it is past k = min(topk, nblocks) or its
 *      block's score is -inf ([CB] docstring: the output is padded with -1; the DCP branch
 *      deselects rows without context only by filling -inf).
 *   R7 DCP local ends: shard d holds the global tokens t < gke with
 *      t % D == d, so its local end is ceil((gke - d) / D) when gke > d,
 *      else 0 ([SG] interleave-1 placement).
 *   R8 masking (below): a logit outside its window or outside the row's
 *      candidate blocks becomes -inf; the rest are untouched.
 *   R12 starts in the DCP form (below, select_sharded_impl): each shard's
 *      window starts at its share of the global start, and blocks count
 *      from there.
 *
 * Floating-point values are widened to double for every comparison; no
 * arithmetic is done on them, so the results are exact.
 */
#include "dsa_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* R4: the total order                                                  */
/* ------------------------------------------------------------------ */

/* Returns <0, 0, >0 as a ranks below, equal to, above b. */
static int total_cmp(double a, double b)
{
    int a_nan = isnan(a) ? 1 : 0;
    int b_nan = isnan(b) ? 1 : 0;
    if (a_nan || b_nan)
        return a_nan - b_nan;
    if (a < b)
        return -1;
    if (a > b)
        return 1;
    /* equal as numbers: only +0 and -0 can still differ; +0 ranks above */
    {
        int a_neg = signbit(a) ? 1 : 0;
        int b_neg = signbit(b) ? 1 : 0;
        return b_neg - a_neg;
    }
}

/* Write a score as fp32; NaN becomes the canonical quiet NaN (R2). */
static float to_score(double v)
{
    if (isnan(v)) {
        uint32_t bits = 0x7FC00000u;
        float f;
        memcpy(&f, &bits, sizeof f);
        return f;
    }
    return (float)v;
}

static int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

/* Python-style floor division for a positive divisor. */
static int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && (a < 0))
        q -= 1;
    return q;
}

/* ------------------------------------------------------------------ */
/* Block scores of one row ([CB] _block_scores_kernel)                  */
/* ------------------------------------------------------------------ */

/*
 * score[b] for b in [0, nb): the maximum (R4) of row[c] over the in-window
 * columns c of block b, i.e. [s + b*bs, s + (b+1)*bs) intersected with
 * [s, e); -inf when that set is empty. With pin and e > s the block
 * (e - s - 1) / bs becomes +inf after the reduction.
 */
static void row_block_scores(const float *row, int64_t s, int64_t e,
                             int64_t bs, int64_t nb, int pin, double *score)
{
    int64_t b, c;
    for (b = 0; b < nb; ++b) {
        int64_t lo = s + b * bs;
        int64_t hi = imin64(lo + bs, e);
        double m = -INFINITY;
        for (c = lo; c < hi; ++c) {
            double x = (double)row[c];
            if (total_cmp(x, m) > 0)
                m = x;
        }
        score[b] = m;
    }
    if (pin && e > s)
        score[(e - s - 1) / bs] = INFINITY;
}

/* Window of row r (R3), with bounds shared by groups of row_repeat rows. */
static void row_window(int64_t r, int64_t width, const int32_t *row_ks,
                       const int32_t *row_ke, int64_t row_repeat,
                       int64_t *s_out, int64_t *e_out)
{
    int64_t g = r / row_repeat;
    int64_t ks = row_ks ? (int64_t)row_ks[g] : 0;
    int64_t ke = (int64_t)row_ke[g];
    int64_t e = imin64(ke, width);
    int64_t s = imin64(imax64(ks, 0), e);
    *s_out = s;
    *e_out = e;
}

/* ------------------------------------------------------------------ */
/* Selection ([CB] scores.topk + _store_candidates_kernel)              */
/* ------------------------------------------------------------------ */

typedef struct {
    double v;
    int32_t id;
} ranked_t;

/* Descending by score (R4), then ascending by id (R5). */
static int ranked_cmp(const void *pa, const void *pb)
{
    const ranked_t *a = (const ranked_t *)pa;
    const ranked_t *b = (const ranked_t *)pb;
    int c = total_cmp(b->v, a->v);
    if (c != 0)
        return c;
    return (a->id > b->id) - (a->id < b->id);
}

/* out[j], j < topk: the j-th ranked block id, or -1 (R6). */
static void select_row(const double *score, int64_t nb, int64_t topk,
                       ranked_t *tmp, int32_t *out)
{
    int64_t b, j;
    int64_t k = imin64(topk, nb);
    for (b = 0; b < nb; ++b) {
        tmp[b].v = score[b];
        tmp[b].id = (int32_t)b;
    }
    qsort(tmp, (size_t)nb, sizeof(ranked_t), ranked_cmp);
    for (j = 0; j < topk; ++j) {
        int keep = j < k && total_cmp(tmp[j].v, -INFINITY) > 0;
        out[j] = keep ? tmp[j].id : -1;
    }
}

/* ------------------------------------------------------------------ */
/* Entry points                                                         */
/* ------------------------------------------------------------------ */

int dsa_oracle_block_scores(const float *logits, int64_t rows, int64_t width,
                            int64_t ld_logits, const int32_t *row_ks,
                            const int32_t *row_ke, int32_t block_size,
                            int32_t row_repeat, int32_t pin_newest,
                            float *scores, int64_t ld_scores)
{
    int64_t r, b, nb;
    double *score;
    if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1)
        return -1;
    if (rows == 0 || width == 0)
        return 0;
    nb = (width + block_size - 1) / block_size;
    score = (double *)malloc((size_t)nb * sizeof(double));
    if (!score)
        return -2;
    for (r = 0; r < rows; ++r) {
        int64_t s, e;
        row_window(r, width, row_ks, row_ke, row_repeat, &s, &e);
        row_block_scores(logits + r * ld_logits, s, e, block_size, nb,
                         pin_newest != 0, score);
        for (b = 0; b < nb; ++b)
            scores[r * ld_scores + b] = to_score(score[b]);
    }
    free(score);
    return 0;
}

int dsa_oracle_select(const float *logits, int64_t rows, int64_t width,
                      int64_t ld_logits, const int32_t *row_ks,
                      const int32_t *row_ke, int32_t topk_blocks,
                      int32_t block_size, int32_t row_repeat,
                      int32_t pin_newest, int32_t *out, int64_t ld_out,
                      float *scores, int64_t ld_scores)
{
    int64_t r, b, j, nb;
    double *score;
    ranked_t *tmp;
    if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1 ||
        topk_blocks < 0)
        return -1;
    if (rows == 0)
        return 0;
    if (width == 0) {
        /* [CB] _select_candidate_blocks_impl: an empty row selects nothing */
        for (r = 0; r < rows; ++r)
            for (j = 0; j < topk_blocks; ++j)
                out[r * ld_out + j] = -1;
        return 0;
    }
    nb = (width + block_size - 1) / block_size;
    score = (double *)malloc((size_t)nb * sizeof(double));
    tmp = (ranked_t *)malloc((size_t)nb * sizeof(ranked_t));
    if (!score || !tmp) {
        free(score);
        free(tmp);
        return -2;
    }
    for (r = 0; r < rows; ++r) {
        int64_t s, e;
        row_window(r, width, row_ks, row_ke, row_repeat, &s, &e);
        row_block_scores(logits + r * ld_logits, s, e, block_size, nb,
                         pin_newest != 0, score);
        if (scores)
            for (b = 0; b < nb; ++b)
                scores[r * ld_scores + b] = to_score(score[b]);
        select_row(score, nb, topk_blocks, tmp, out + r * ld_out);
    }
    free(score);
    free(tmp);
    return 0;
}

/*
 * [CB] _select_candidate_blocks_impl, DCP branch, with the shards held as a
 * leading axis: logits is [shards, rows, local_width] (shard stride
 * shard_stride, row stride ld_logits). For each row:
 *   1. per shard d, local block scores with pin off, local block size
 *      gbs / shards, local start 0 and local end ceil((gke - d) / shards)
 *      when gke > d, else 0 (R7), clamped to local_width;
 *   2. G[b] = max over shards of the local scores, for
 *      b < min(ceil(local_width / lbs), nbg), -inf beyond; nbg =
 *      max(max_global_blocks, 1);
 *   3. G[clamp((gke - 1) // gbs, 0, nbg - 1)] = +inf;
 *   4. gke <= 0 makes every G[b] = -inf;
 *   5. selection with k = min(topk, nbg).
 */
/*
 * R12 (starts in the DCP form; the pages' DCP branch has no starts and pins
 * (ends - 1) // gbs, which is this rule with a start of 0): a row's global
 * window is [gs, ge) with ge = gke and gs = min(max(gks, 0), max(gke, 0)).
 * Shard d holds the global tokens t with t % shards == d, so its window is
 * local columns [ceil((gs - d) / shards), ceil((ge - d) / shards)) (each 0
 * when the global bound is <= d), clamped to local_width. Global blocks are
 * request-local (R1): block b covers tokens [gs + b*gbs, gs + (b+1)*gbs),
 * and shard d's share of it is local block b counted from the shard's own
 * window start. The pin is block (ge - gs - 1) // gbs, clamped to nbg - 1,
 * and a row with ge <= gs selects nothing. Without starts (gks = 0) this is
 * exactly steps 1-5 above.
 */
static int select_sharded_impl(const float *logits, int32_t shards, int64_t rows,
                               int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                               const int32_t *global_row_ks, const int32_t *global_row_ke,
                               int32_t global_block_size, int32_t max_global_blocks,
                               int32_t row_repeat, int32_t topk_blocks, int32_t *out,
                               int64_t ld_out, float *scores, int64_t ld_scores)
{
    int64_t r, b, d, nbg, lbs, nlb, n_use;
    double *global_score, *local_score;
    ranked_t *tmp;
    if (shards < 1 || rows < 0 || local_width < 0 || global_block_size < 1 ||
        global_block_size % shards != 0 || row_repeat < 1 || topk_blocks < 0)
        return -1;
    if (rows == 0)
        return 0;
    nbg = max_global_blocks > 1 ? max_global_blocks : 1;
    lbs = global_block_size / shards;
    nlb = (local_width + lbs - 1) / lbs;
    n_use = imin64(nlb, nbg);
    global_score = (double *)malloc((size_t)nbg * sizeof(double));
    local_score = (double *)malloc((size_t)(nlb > 0 ? nlb : 1) * sizeof(double));
    tmp = (ranked_t *)malloc((size_t)nbg * sizeof(ranked_t));
    if (!global_score || !local_score || !tmp) {
        free(global_score);
        free(local_score);
        free(tmp);
        return -2;
    }
    for (r = 0; r < rows; ++r) {
        int64_t gke = (int64_t)global_row_ke[r / row_repeat];
        int64_t gks = global_row_ks ? (int64_t)global_row_ks[r / row_repeat] : 0;
        int64_t gs = imin64(imax64(gks, 0), imax64(gke, 0));
        int64_t pin;
        for (b = 0; b < nbg; ++b)
            global_score[b] = -INFINITY;
        for (d = 0; d < shards; ++d) {
            const float *row = logits + d * shard_stride + r * ld_logits;
            int64_t lks = gs > d ? (gs - d + shards - 1) / shards : 0;
            int64_t lke = gke > d ? (gke - d + shards - 1) / shards : 0;
            int64_t e = imin64(lke, local_width);
            int64_t s = imin64(lks, e);
            if (nlb == 0)
                continue;
            row_block_scores(row, s, e, lbs, nlb, 0, local_score);
            for (b = 0; b < n_use; ++b)
                if (total_cmp(local_score[b], global_score[b]) > 0)
                    global_score[b] = local_score[b];
        }
        pin = floor_div(gke - gs - 1, global_block_size);
        pin = imin64(imax64(pin, 0), nbg - 1);
        global_score[pin] = INFINITY;
        if (gke <= gs)
            for (b = 0; b < nbg; ++b)
                global_score[b] = -INFINITY;
        if (scores)
            for (b = 0; b < nbg; ++b)
                scores[r * ld_scores + b] = to_score(global_score[b]);
        select_row(global_score, nbg, topk_blocks, tmp, out + r * ld_out);
    }
    free(global_score);
    free(local_score);
    free(tmp);
    return 0;
}

int dsa_oracle_select_sharded(const float *logits, int32_t shards,
                              int64_t rows, int64_t local_width,
                              int64_t ld_logits, int64_t shard_stride,
                              const int32_t *global_row_ke,
                              int32_t global_block_size,
                              int32_t max_global_blocks, int32_t row_repeat,
                              int32_t topk_blocks, int32_t *out,
                              int64_t ld_out, float *scores, int64_t ld_scores)
{
    return select_sharded_impl(logits, shards, rows, local_width, ld_logits, shard_stride,
                               NULL, global_row_ke, global_block_size, max_global_blocks,
                               row_repeat, topk_blocks, out, ld_out, scores, ld_scores);
}

int dsa_oracle_select_sharded_starts(const float *logits, int32_t shards, int64_t rows,
                                     int64_t local_width, int64_t ld_logits,
                                     int64_t shard_stride, const int32_t *global_row_ks,
                                     const int32_t *global_row_ke, int32_t global_block_size,
                                     int32_t max_global_blocks, int32_t row_repeat,
                                     int32_t topk_blocks, int32_t *out, int64_t ld_out,
                                     float *scores, int64_t ld_scores)
{
    return select_sharded_impl(logits, shards, rows, local_width, ld_logits, shard_stride,
                               global_row_ks, global_row_ke, global_block_size,
                               max_global_blocks, row_repeat, topk_blocks, out, ld_out, scores,
                               ld_scores);
}

/* ------------------------------------------------------------------ */
/* Masking to candidates ([CB] masking function after selection)        */
/* ------------------------------------------------------------------ */

/*
 * R8 (reading of the masking function, whose body is not on the page): in
 * place, logits[r][c] for c in [0, width) becomes -inf when c lies outside the
 * row's window [s, e) (R3) or when its request-local block (c - s) / bs is
 * not one of the row's candidate ids cand[r][0 .. topk) (ids < 0 are empty
 * slots). Kept logits are left bit for bit as they were.
 */
static int is_candidate(const int32_t *cand, int64_t topk, int64_t b)
{
    int64_t j;
    for (j = 0; j < topk; ++j)
        if (cand[j] >= 0 && (int64_t)cand[j] == b)
            return 1;
    return 0;
}

int dsa_oracle_mask(float *logits, int64_t rows, int64_t width, int64_t ld_logits,
                    const int32_t *row_ks, const int32_t *row_ke,
                    const int32_t *cand, int64_t topk, int64_t ld_cand,
                    int32_t block_size, int32_t row_repeat)
{
    int64_t r, c;
    if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1 || topk < 0)
        return -1;
    for (r = 0; r < rows; ++r) {
        int64_t s, e;
        float *row = logits + r * ld_logits;
        row_window(r, width, row_ks, row_ke, row_repeat, &s, &e);
        for (c = 0; c < width; ++c) {
            int keep = c >= s && c < e &&
                       is_candidate(cand + r * ld_cand, topk, (c - s) / block_size);
            if (!keep)
                row[c] = -INFINITY;
        }
    }
    return 0;
}

/*
 * The DCP form: shard d of row r keeps its local columns [0, lke_d) (R7)
 * whose local block c / (gbs / shards) is a candidate of the row; the
 * candidate ids are global block ids, which name the same local blocks on
 * every shard ([CB] masking function: under DCP the local block size is
 * passed and the ids apply unchanged).
 */
static int mask_sharded_impl(float *logits, int32_t shards, int64_t rows,
                             int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                             const int32_t *global_row_ks, const int32_t *global_row_ke,
                             int32_t global_block_size, int32_t row_repeat,
                             const int32_t *cand, int64_t topk, int64_t ld_cand)
{
    int64_t r, d, c, lbs;
    if (shards < 1 || rows < 0 || local_width < 0 || global_block_size < 1 ||
        global_block_size % shards != 0 || row_repeat < 1 || topk < 0)
        return -1;
    lbs = global_block_size / shards;
    for (r = 0; r < rows; ++r) {
        int64_t gke = (int64_t)global_row_ke[r / row_repeat];
        int64_t gks = global_row_ks ? (int64_t)global_row_ks[r / row_repeat] : 0;
        int64_t gs = imin64(imax64(gks, 0), imax64(gke, 0));
        for (d = 0; d < shards; ++d) {
            float *row = logits + d * shard_stride + r * ld_logits;
            int64_t lks = gs > d ? (gs - d + shards - 1) / shards : 0;
            int64_t lke = gke > d ? (gke - d + shards - 1) / shards : 0;
            int64_t e = imin64(lke, local_width);
            int64_t s = imin64(lks, e);
            for (c = 0; c < local_width; ++c) {
                int keep = c >= s && c < e &&
                           is_candidate(cand + r * ld_cand, topk, (c - s) / lbs);
                if (!keep)
                    row[c] = -INFINITY;
            }
        }
    }
    return 0;
}

int dsa_oracle_mask_sharded(float *logits, int32_t shards, int64_t rows, int64_t local_width,
                            int64_t ld_logits, int64_t shard_stride,
                            const int32_t *global_row_ke, int32_t global_block_size,
                            int32_t row_repeat, const int32_t *cand, int64_t topk,
                            int64_t ld_cand)
{
    return mask_sharded_impl(logits, shards, rows, local_width, ld_logits, shard_stride, NULL,
                             global_row_ke, global_block_size, row_repeat, cand, topk,
                             ld_cand);
}

/* The DCP masking with starts (R12): shard d keeps the candidate blocks of
 * its own window [ceil((gs - d) / shards), ceil((ge - d) / shards)), local
 * blocks counted from that window's start. */
int dsa_oracle_mask_sharded_starts(float *logits, int32_t shards, int64_t rows,
                                   int64_t local_width, int64_t ld_logits,
                                   int64_t shard_stride, const int32_t *global_row_ks,
                                   const int32_t *global_row_ke, int32_t global_block_size,
                                   int32_t row_repeat, const int32_t *cand, int64_t topk,
                                   int64_t ld_cand)
{
    return mask_sharded_impl(logits, shards, rows, local_width, ld_logits, shard_stride,
                             global_row_ks, global_row_ke, global_block_size, row_repeat, cand,
                             topk, ld_cand);
}
