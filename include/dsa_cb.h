/*
 * dsa_cb.h -- C ABI of the GB300 (sm_103a) DSA candidate-block selection
 * library (libdsa_cb.so).
 *
 * The operation: every indexer-logit row is masked to its window
 * [row_ks, row_ke) in packed column space, max-reduced per block of
 * block_size columns counted from the window start, optionally has its newest
 * block pinned to +inf, and yields the ids of its top topk_blocks blocks,
 * -1 padded. Source: the page "launcher/dcp2/diffs/02-model_executor_
 * kernels_attention_dsa_candidate_blocks.py.diff" (vLLM-fork
 * candidate_blocks.py): _max_with_nan, _block_scores_kernel, _block_scores,
 * select_candidate_blocks / _select_candidate_blocks_impl and the
 * _store_candidates_kernel launch. The DCP form takes the interleave-1 token
 * placement of the page "sgl-project--sglang/python/sglang/srt/layers/dcp/
 * kernels.py" (create_triton_kv_indices_for_dcp_triton).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named logits, row_ks, row_ke, global_row_ke, out, scores_out
 *    and workspace are DEVICE addresses of memory owned by the caller:
 *    device memory, or page-locked host memory under the address that
 *    dsa_mapped_host_pointer gives (the kernels then read and write it
 *    across the host link). The library allocates no memory and keeps no
 *    pointer after a call returns.
 *  - Matrices are row-major with an explicit row stride in elements (ld_*).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL means the legacy
 *    default stream) and the call returns without synchronising. Results are
 *    ready when the stream reaches that point.
 *  - Bounds are int32 and shared by groups of row_repeat consecutive rows:
 *    row r reads entry r / row_repeat, so row_ks and row_ke hold
 *    ceil(rows / row_repeat) entries.
 *  - Out-of-range bounds are clamped, never trapped: e = min(ke, width),
 *    s = min(max(ks, 0), e); a window with s >= e is empty.
 *  - Block scores are fp32. Any NaN in a block makes its score the canonical
 *    quiet NaN 0x7FC00000. Scores are ranked in the total order
 *    -inf < ... < -0 < +0 < ... < +inf < NaN; equal scores rank the lower
 *    block id first. A slot whose block scores -inf, or which lies past
 *    k = min(topk_blocks, number of blocks), holds -1.
 *  - Return values: DSA_OK, or an error code. Argument errors are detected
 *    on the host before anything is enqueued. No entry point traps or spins
 *    on the device.
 */
#ifndef DSA_CB_H
#define DSA_CB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_EINVAL = -1,       /* invalid argument; nothing was enqueued         */
    DSA_ECUDA = -2,        /* a CUDA runtime call or kernel launch failed    */
    DSA_EUNSUPPORTED = -3  /* valid, but beyond this build's limits (below)  */
} dsa_status;

/* Static text for a status code (never NULL). */
const char *dsa_status_string(int status);

/* Largest number of blocks per row that the selecting entry points accept
 * (all block scores of a row are kept in on-chip shared memory while its
 * top-k is taken). Larger rows return DSA_EUNSUPPORTED. */
int32_t dsa_select_max_blocks(void);

/* Largest shard count accepted by dsa_select_candidate_blocks_sharded. */
int32_t dsa_select_max_shards(void);

/*
 * Bytes of optional device workspace that lets the selecting entry points
 * deal rows to CTAs as they free up and split long rows over several CTAs:
 * a 256-byte header (a work counter and a count of finished CTAs), one
 * arrival counter per row, then rows * nblocks block keys, each part
 * 256-byte aligned. nblocks is ceil(width / block_size) for
 * dsa_select_candidate_blocks and max(max_global_blocks, 1) for the sharded
 * form. Returns 0 for negative arguments and for rows == 0.
 *
 * Workspace contract: caller-owned device memory of at least this many bytes,
 * all zero bytes before its first use (e.g. one cudaMemset), and written by
 * nothing but these calls afterwards. Every completed call leaves its header
 * and counters at zero; block keys that a call of another shape left where
 * this call's counters are can never be mistaken for a count, so one
 * workspace serves calls of any shape in turn. Two calls that may run at the
 * same time (different streams) must not share a workspace.
 */
size_t dsa_select_workspace_bytes(int64_t rows, int64_t nblocks);

/*
 * dsa_select_set_launch_override -- pins one launch-shape choice of the
 * selecting entry points for every later call in this process, or hands it
 * back to the launcher (value 0). The pages have no counterpart: the
 * launcher picks a shape from each call's sizes, results never depend on
 * the shape (only the speed does), and tests and tuning sweeps use this to
 * run shapes that the automatic choice reaches only at other sizes. Normal
 * callers never need it. The setting is process-wide; set it while no other
 * host thread is issuing selecting calls.
 *
 *   DSA_LAUNCH_SPLIT       CTAs per row when a workspace is given, 1..8
 *   DSA_LAUNCH_THREADS     threads per row-per-CTA block, 128 or 256
 *   DSA_LAUNCH_WARP_ROWS   1: never take the one-row-per-warp kernel
 *   DSA_LAUNCH_WARP_ORDER  1: one-row-per-warp rows in order (default: last
 *                          to first)
 *   DSA_LAUNCH_PIPELINE    0 (automatic): the pipelined (bulk-copy staged)
 *                          kernels take the unsharded calls they support, the
 *                          DCP forms stay on the row-per-CTA kernel; 1: never
 *                          take the pipelined kernels; 2: take them (DCP
 *                          forms included) with every warp on one row; 3:
 *                          take them with one row per warp (unsharded rows
 *                          with top-k <= 32 and <= 2048 blocks)
 *   DSA_LAUNCH_PIPE_SPLIT  pipelined kernels: parts per row, 1..8 (only
 *                          with a workspace)
 *   DSA_LAUNCH_PIPE_STAGES pipelined kernels: ring depth, 2..16
 *   DSA_LAUNCH_PIPE_STAGE_KB  pipelined kernels: KiB per stage, 4..64
 *   DSA_LAUNCH_PIPE_SCHED  pipelined kernels: 1 = rows dealt to CTAs in a
 *                          fixed order even when a workspace is given
 *   DSA_LAUNCH_PIPE_WARPS  pipelined kernels, every warp on one row: 4 or 8
 *                          consumer warps per CTA (default: 8, one CTA per
 *                          SM, for rows of more than 256 KiB; else 4)
 *   DSA_LAUNCH_PIPE_CTAS   pipelined kernels: CTAs per SM, 1..4 (at most 2
 *                          with 8 consumer warps or one row per warp)
 *   DSA_LAUNCH_PIPE_STAGE_OWNER  pipelined kernels, every warp on one row:
 *                          1 = each folding warp takes whole stages in turn
 *                          (default: every stage's blocks shared by all)
 *   DSA_LAUNCH_PIPE_ORDER  pipelined kernels, every warp on one row: 1 = rows
 *                          handed out in index order (the default), 2 =
 *                          longest rows first whenever the call allows it,
 *                          3 = index order with each CTA's next rows claimed
 *                          ahead from the start (not as it frees up)
 *   DSA_LAUNCH_RANK_CTA    row-per-CTA kernel: 1 = every warp of the CTA
 *                          ranks each row, 2 = one warp ranks every row of
 *                          up to 1024 live blocks with k <= 32 (default: one
 *                          warp, except the fp32 DCP form without starts);
 *                          pipelined kernel: 2 = one rank warp ranks rows
 *                          of up to 1024 live blocks with k <= 32 (default:
 *                          all four rank warps)
 *
 * DSA_EINVAL for an unknown knob or a value outside its range (nothing
 * changes then).
 */
enum {
    DSA_LAUNCH_SPLIT = 1,
    DSA_LAUNCH_THREADS = 2,
    DSA_LAUNCH_WARP_ROWS = 3,
    DSA_LAUNCH_WARP_ORDER = 4,
    DSA_LAUNCH_PIPELINE = 5,
    DSA_LAUNCH_PIPE_SPLIT = 6,
    DSA_LAUNCH_PIPE_STAGES = 7,
    DSA_LAUNCH_PIPE_STAGE_KB = 8,
    DSA_LAUNCH_PIPE_SCHED = 9,
    DSA_LAUNCH_PIPE_WARPS = 10,
    DSA_LAUNCH_PIPE_CTAS = 11,
    DSA_LAUNCH_PIPE_STAGE_OWNER = 12,
    DSA_LAUNCH_PIPE_ORDER = 13,
    DSA_LAUNCH_RANK_CTA = 14
};
dsa_status dsa_select_set_launch_override(int32_t knob, int32_t value);

/*
 * dsa_pipeline_error -- whether a pipelined selecting kernel has given up a
 * wait since the process started (or since the last clear). The pages have
 * no counterpart. The pipelined kernels stage logits through shared memory
 * with the bulk-copy engine and wait on mbarriers; every such wait ends
 * after one second, records a nonzero site code in a device-wide flag and
 * lets the kernel finish instead of hanging the GPU. Such a call's outputs
 * are not valid. Returns that flag (0: no wait ever gave up; 1: a consumer's
 * wait for data; 2: the producer's wait for a free stage), or -1 if the flag
 * could not be read. clear != 0 resets it to 0 after reading. Synchronises
 * with the current device (a plain device-to-host copy of 4 bytes).
 */
int dsa_pipeline_error(int clear);

/*
 * dsa_block_scores -- per-block scores of every row (candidate_blocks.py:
 * _block_scores and _block_scores_kernel, with the PIN_NEWEST switch).
 *
 *   logits      [rows, ld_logits] fp32; columns [0, width) are read.
 *   row_ks      nullable; NULL means every window starts at 0.
 *   row_ke      window ends, ceil(rows / row_repeat) entries.
 *   block_size  >= 1; nb = ceil(width / block_size) blocks per row.
 *   pin_newest  nonzero: when e > s, block (e - s - 1) / block_size of the
 *               row becomes +inf after the reduction.
 *   scores_out  [rows, ld_scores] fp32, ld_scores >= nb; entry (r, b) is
 *               the max over the in-window columns
 *               [s + b*block_size, s + (b+1)*block_size) and [s, e), or
 *               -inf when that set is empty.
 *
 * rows == 0 or width == 0: DSA_OK, nothing written. DSA_EINVAL for
 * rows < 0, width < 0, block_size < 1, row_repeat < 1, ld_logits < width,
 * ld_scores < nb, or a NULL logits / row_ke / scores_out. DSA_EUNSUPPORTED
 * for width >= 2^31.
 */
dsa_status dsa_block_scores(const float *logits, int64_t rows, int64_t width,
                            int64_t ld_logits, const int32_t *row_ks,
                            const int32_t *row_ke, int32_t block_size,
                            int32_t row_repeat, int32_t pin_newest,
                            float *scores_out, int64_t ld_scores,
                            void *stream);

/*
 * dsa_select_candidate_blocks -- ranked candidate block ids per row
 * (candidate_blocks.py: select_candidate_blocks / _select_candidate_blocks_impl
 * without a DCP group: block scores, then top-k, then the -1-padded store).
 * The pages always pin the newest block here; pin_newest exposes the switch.
 *
 *   out         [rows, ld_out] int32, ld_out >= topk_blocks; slot j < topk
 *               holds the block id of rank j (rank by score, then lower id)
 *               or -1 (see the conventions above). Slots >= topk_blocks of
 *               each row are left untouched.
 *   scores_out  nullable; when given, [rows, ld_scores] fp32 with
 *               ld_scores >= nb receives the block scores that were ranked
 *               (pin applied), as dsa_block_scores would write them.
 *   workspace   nullable; see dsa_select_workspace_bytes. With a workspace
 *               of sufficient size rows are dealt to CTAs as they free up
 *               and long rows are split over several CTAs (their block keys
 *               meet in the workspace and the last CTA of the row to finish
 *               ranks them); without one, rows are dealt in a fixed order
 *               and none is split. Results are identical either way.
 *
 * rows == 0: DSA_OK, nothing written. width == 0: every slot of out is -1.
 * topk_blocks == 0 and no scores_out: DSA_OK, nothing written. A workspace
 * smaller than dsa_select_workspace_bytes is not used.
 * DSA_EINVAL for negative rows / width / topk_blocks, block_size < 1,
 * row_repeat < 1, ld_logits < width, ld_out < topk_blocks, ld_scores < nb
 * (with scores_out), or a NULL logits / row_ke / out (out only when
 * topk_blocks > 0). DSA_EUNSUPPORTED when nb > dsa_select_max_blocks(),
 * width > 2^31 - 8193 or rows > 2^28 - 1.
 */
dsa_status dsa_select_candidate_blocks(const float *logits, int64_t rows,
                                       int64_t width, int64_t ld_logits,
                                       const int32_t *row_ks,
                                       const int32_t *row_ke,
                                       int32_t topk_blocks, int32_t block_size,
                                       int32_t row_repeat, int32_t pin_newest,
                                       int32_t *out, int64_t ld_out,
                                       float *scores_out, int64_t ld_scores,
                                       void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * dsa_select_candidate_blocks_sharded -- the DCP form on one device
 * (candidate_blocks.py: _select_candidate_blocks_impl with a DCP group), the
 * D ranks' local logits held as a leading axis instead of on D GPUs.
 *
 *   logits         shard d, row r, local column c at
 *                  logits[d * shard_stride + r * ld_logits + c], c <
 *                  local_width; local column c of shard d is global token
 *                  shards * c + d (interleave 1).
 *   global_row_ke  global window end of each row group (no starts: every
 *                  global window begins at token 0).
 *   global_block_size  multiple of shards; the local block is
 *                  global_block_size / shards columns, so local block b of
 *                  every shard is its share of global block b.
 *   max_global_blocks  number of global blocks nbg = max(value, 1); ids are
 *                  in [0, nbg).
 *   out, scores_out, workspace  as for dsa_select_candidate_blocks with
 *                  nb = nbg.
 *
 * Per row: shard d's window is its first ceil((gke - d) / shards) local
 * columns when gke > d (else empty), clamped to local_width; local block
 * scores are taken without a pin; the global score of block b is the max
 * over shards for b < min(ceil(local_width / local block), nbg) and -inf
 * beyond; block clamp((gke - 1) // global_block_size, 0, nbg - 1) becomes
 * +inf; a row with gke <= 0 scores -inf everywhere; then top-k and -1 as
 * above.
 *
 * rows == 0: DSA_OK. DSA_EINVAL for shards < 1, negative rows / local_width
 * / topk_blocks, global_block_size < 1 or not a multiple of shards,
 * row_repeat < 1, ld_logits < local_width, shard_stride < 0, ld_out <
 * topk_blocks, ld_scores < nbg (with scores_out), or a NULL
 * global_row_ke / out (out only when topk_blocks > 0) / logits (when
 * local_width > 0). DSA_EUNSUPPORTED when nbg > dsa_select_max_blocks(),
 * shards > dsa_select_max_shards(), local_width > 2^31 - 8193 or
 * rows > 2^28 - 1.
 */
dsa_status dsa_select_candidate_blocks_sharded(
    const float *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ke,
    int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
    int32_t topk_blocks, int32_t *out, int64_t ld_out, float *scores_out,
    int64_t ld_scores, void *workspace, size_t workspace_bytes, void *stream);

/*
 * dsa_mask_candidate_logits -- mask packed logits to the selected candidate
 * blocks, in place (candidate_blocks.py: the masking function after
 * selection, whose docstring masks logits outside the causal window or
 * outside the request-local candidate blocks; its body is not on the page).
 *
 *   logits       [rows, ld_logits] fp32, modified in place over columns
 *                [0, width): column c becomes -inf when it lies outside the
 *                row's window [s, e) (clamped as for selection) or when its
 *                request-local block (c - s) / block_size is not among
 *                candidates[r, 0 .. topk_blocks); entries < 0 are empty
 *                slots. Kept columns are not read or written.
 *   candidates   [rows, ld_candidates] int32, e.g. the `out` of
 *                dsa_select_candidate_blocks; nullable when topk_blocks == 0
 *                (then every column is masked).
 *   row_ks, row_ke, block_size, row_repeat  as for the selection.
 *
 * rows == 0 or width == 0: DSA_OK, nothing written. DSA_EINVAL for negative
 * rows / width / topk_blocks, block_size < 1, row_repeat < 1, ld_logits <
 * width, ld_candidates < topk_blocks, or a NULL logits / row_ke / candidates
 * (candidates only when topk_blocks > 0). DSA_EUNSUPPORTED for widths near
 * 2^31.
 */
dsa_status dsa_mask_candidate_logits(float *logits, int64_t rows, int64_t width,
                                     int64_t ld_logits, const int32_t *row_ks,
                                     const int32_t *row_ke,
                                     const int32_t *candidates,
                                     int32_t topk_blocks, int64_t ld_candidates,
                                     int32_t block_size, int32_t row_repeat,
                                     void *stream);

/*
 * dsa_mask_candidate_logits_sharded -- the DCP form of the masking: shard d of
 * row r keeps its local columns below ceil((gke - d) / shards) (none when
 * gke <= d) whose local block c / (global_block_size / shards) is a
 * candidate; the candidate ids are global block ids, which name the same
 * local blocks on every shard. Layout, strides and errors as for
 * dsa_select_candidate_blocks_sharded and dsa_mask_candidate_logits.
 */
dsa_status dsa_mask_candidate_logits_sharded(
    float *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ke,
    int32_t global_block_size, int32_t row_repeat, const int32_t *candidates,
    int32_t topk_blocks, int64_t ld_candidates, void *stream);

/*
 * dsa_select_candidate_blocks_sharded_starts -- the DCP form with global
 * window starts (the pages' DCP branch has none; its pin (ends - 1) // gbs is
 * the start-0 case of the rule below). Row r's global window is [gs, ge)
 * with ge = global_row_ke[r / row_repeat] and gs = min(max(global_row_ks[...],
 * 0), max(ge, 0)). Shard d holds the global tokens t with t % shards == d,
 * so its window is local columns [ceil((gs - d) / shards),
 * ceil((ge - d) / shards)) (0 when the bound is <= d), clamped to
 * local_width. Global blocks are request-local: block b covers tokens
 * [gs + b*gbs, gs + (b+1)*gbs), which is local block b of every shard counted
 * from the shard's own window start. The pin is block
 * min((ge - gs - 1) // gbs, nbg - 1); a row with ge <= gs selects nothing.
 * Local blocks past min(ceil(local_width / lbs), nbg) are dropped as in the
 * form without starts. A NULL global_row_ks is the form without starts.
 * Every other argument, limit and error is that of
 * dsa_select_candidate_blocks_sharded. Each shard row is streamed on its own
 * (its start sets its alignment), so rows with starts take a slightly slower
 * path than rows without.
 */
dsa_status dsa_select_candidate_blocks_sharded_starts(
    const float *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ks,
    const int32_t *global_row_ke, int32_t global_block_size,
    int32_t max_global_blocks, int32_t row_repeat, int32_t topk_blocks,
    int32_t *out, int64_t ld_out, float *scores_out, int64_t ld_scores,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * dsa_mask_candidate_logits_sharded_starts -- the DCP masking with global
 * window starts: shard d keeps the columns of its window (as above) whose
 * local block, counted from the shard's window start, is a candidate.
 * Arguments and errors as for dsa_mask_candidate_logits_sharded, plus the
 * nullable global_row_ks.
 */
dsa_status dsa_mask_candidate_logits_sharded_starts(
    float *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ks,
    const int32_t *global_row_ke, int32_t global_block_size, int32_t row_repeat,
    const int32_t *candidates, int32_t topk_blocks, int64_t ld_candidates,
    void *stream);

/*
 * bf16 logits. The same operations on bf16 logits, held as their 16-bit
 * patterns (uint16_t, the layout of torch.bfloat16 / __nv_bfloat16). The page
 * allocates the block scores with the logits' dtype (_block_scores:
 * logits.new_empty), so scores_out is bf16 too: a block score is the
 * block's max bf16 value (exact), +inf / -inf (0x7F80 / 0xFF80), or the
 * canonical bf16 NaN 0x7FC0. Masking writes bf16 -inf (0xFF80). Selection
 * ranks the exact values, so a bf16 call gives the same ids as the fp32 call
 * on the widened logits. Arguments (in elements), limits and errors are
 * those of the fp32 entry points above; the vectorised paths need the row
 * starts to be 16-byte (8-element) aligned as before, and fall back to
 * 8-, 4- or 2-byte loads otherwise.
 */
dsa_status dsa_block_scores_bf16(const uint16_t *logits, int64_t rows, int64_t width,
                                 int64_t ld_logits, const int32_t *row_ks,
                                 const int32_t *row_ke, int32_t block_size,
                                 int32_t row_repeat, int32_t pin_newest,
                                 uint16_t *scores_out, int64_t ld_scores, void *stream);

dsa_status dsa_select_candidate_blocks_bf16(
    const uint16_t *logits, int64_t rows, int64_t width, int64_t ld_logits,
    const int32_t *row_ks, const int32_t *row_ke, int32_t topk_blocks,
    int32_t block_size, int32_t row_repeat, int32_t pin_newest, int32_t *out,
    int64_t ld_out, uint16_t *scores_out, int64_t ld_scores, void *workspace,
    size_t workspace_bytes, void *stream);

dsa_status dsa_select_candidate_blocks_sharded_bf16(
    const uint16_t *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ke,
    int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
    int32_t topk_blocks, int32_t *out, int64_t ld_out, uint16_t *scores_out,
    int64_t ld_scores, void *workspace, size_t workspace_bytes, void *stream);

dsa_status dsa_mask_candidate_logits_bf16(uint16_t *logits, int64_t rows, int64_t width,
                                          int64_t ld_logits, const int32_t *row_ks,
                                          const int32_t *row_ke,
                                          const int32_t *candidates,
                                          int32_t topk_blocks, int64_t ld_candidates,
                                          int32_t block_size, int32_t row_repeat,
                                          void *stream);

dsa_status dsa_mask_candidate_logits_sharded_bf16(
    uint16_t *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ke,
    int32_t global_block_size, int32_t row_repeat, const int32_t *candidates,
    int32_t topk_blocks, int64_t ld_candidates, void *stream);

dsa_status dsa_select_candidate_blocks_sharded_starts_bf16(
    const uint16_t *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ks,
    const int32_t *global_row_ke, int32_t global_block_size,
    int32_t max_global_blocks, int32_t row_repeat, int32_t topk_blocks,
    int32_t *out, int64_t ld_out, uint16_t *scores_out, int64_t ld_scores,
    void *workspace, size_t workspace_bytes, void *stream);

dsa_status dsa_mask_candidate_logits_sharded_starts_bf16(
    uint16_t *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ks,
    const int32_t *global_row_ke, int32_t global_block_size, int32_t row_repeat,
    const int32_t *candidates, int32_t topk_blocks, int64_t ld_candidates,
    void *stream);

/*
 * dsa_select_candidate_blocks_sharded_static -- dsa_select_candidate_blocks_
 * sharded without a caller-supplied workspace. The pages have no counterpart:
 * this entry point exists for callers that must not allocate device memory
 * when they call, such as serving engines whose memory planner reserves
 * nearly all of HBM at start-up (a cudaMalloc in the middle of a step could
 * fail or stall on the allocator) and plugin hosts whose operators may not
 * allocate on their own.
 *
 * It allocates nothing. Its workspace is a fixed 8 MiB array that the library
 * declares in device memory; every GPU that loads the library holds that
 * array until the process exits, and all calls on a GPU share it.
 *
 *   Arguments, results and errors are those of
 *   dsa_select_candidate_blocks_sharded (without workspace and
 *   workspace_bytes); every argument error is returned before anything is
 *   enqueued. When dsa_select_workspace_bytes(rows, max(max_global_blocks,
 *   1)) is at most 8 MiB (8388608 bytes) the call uses the array as its
 *   workspace; above that it runs without a workspace (rows dealt to CTAs
 *   in a fixed order, none split), with the same results. Row counts beyond
 *   the selecting calls' limit (2^28 - 1) return DSA_EUNSUPPORTED.
 *
 * Each call that uses the array looks up its device address with
 * cudaGetSymbolAddress, with the call's device current; the first such call
 * on a device may load the library's device code there, so make it before
 * any stream capture. Each such call clears the array's header and arrival
 * counters with cudaMemsetAsync on `stream`. Calls that overlap on the GPU
 * (different streams, or different host threads) race on the shared array
 * and must not be issued.
 */
dsa_status dsa_select_candidate_blocks_sharded_static(
    const float *logits, int32_t shards, int64_t rows, int64_t local_width,
    int64_t ld_logits, int64_t shard_stride, const int32_t *global_row_ke,
    int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
    int32_t topk_blocks, int32_t *out, int64_t ld_out, float *scores_out,
    int64_t ld_scores, void *stream);

/*
 * dsa_mapped_host_pointer -- the device address of page-locked host memory.
 * The pages have no counterpart: it lets a caller whose logits sit in host
 * memory hand them to the selecting, scoring and masking entry points
 * without copying the tensor to the device first. Page-locked memory
 * (cudaHostAlloc / cudaMallocHost, cudaHostRegister, a pinned torch tensor)
 * is mapped into every device's address space; on Grace systems the GPU
 * reads it across NVLink-C2C, so a selecting call reads only the in-window
 * logits across the link instead of the caller copying the whole tensor.
 *
 *   host    a pointer into page-locked host memory (any offset).
 *   device  receives the address under which the current device's kernels
 *           read and write the same bytes.
 *
 * Nothing is launched. DSA_EINVAL when host or device is NULL, or when host
 * is not page-locked memory mapped for the current device (pageable and
 * device memory included); *device is then unchanged. The memory stays the
 * caller's: it must stay allocated and page-locked until the calls that use
 * the address have finished on the GPU.
 */
dsa_status dsa_mapped_host_pointer(const void *host, void **device);

#ifdef __cplusplus
}
#endif

#endif /* DSA_CB_H */
