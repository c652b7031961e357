// dsa_cb.cu -- sm_103a kernels and the C ABI of include/dsa_cb.h.
//
// One pass over HBM per call: every in-window logit is read once, block keys
// stay in shared memory, the top-k runs on them in place, and only ids (and,
// on request, block scores) are written back.
//
// Selecting kernel (select_kernel): up to `split` CTAs per row (1 without a
// workspace). The row's blocks that hold in-window data are cut from its
// start into parts of `chunk` blocks (whole units of 32 blocks), launched
// chunk-major, and a row uses only the parts its data reaches; each CTA
// streams its part (stream.cuh) into a shared-memory key array. A row held
// by one CTA is then pinned, its scores written if asked, and ranked
// (topk.cuh) in place. Otherwise every CTA of the row publishes its keys to
// the row's slice of the workspace and counts itself in on the row's counter
// (arrive_units); the last CTA to arrive reads the other parts back (they
// are in L2) and runs the pin and the top-k. The others exit as soon as they
// have published, so their slots go back to streaming. The DCP form is the same kernel reading `shards` slices per row
// and taking the max over them before the reduction, i.e. the all-reduce MAX
// of candidate_blocks.py's DCP branch happens in registers.
//
// Scores-only kernel (block_scores_kernel): one CTA per (row, chunk of
// blocks), no top-k.
#include "../../include/dsa_cb.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "keys.cuh"
#include "select_pipe.h"
#include "stream.cuh"
#include "topk.cuh"
#include "topk_warp.cuh"

namespace dsa {
namespace {

constexpr int32_t kMaxSelectBlocks = 16384;
constexpr int32_t kMaxShards = 1024;
constexpr int32_t kSplitUnit = 32;  // blocks per unit of a row split
constexpr int kMaxSplit = 8;        // CTAs per row at most
constexpr int kThreads = 256;       // scores-only kernel

// Row layouts of select_kernel.
constexpr int kUnsharded = 0;       // [rows, ld], window [ks, ke)
constexpr int kSharded = 1;         // [shards, rows, ld], windows from 0 (the pages' DCP form)
constexpr int kShardedStarts = 2;   // [shards, rows, ld], windows from each shard's start

// A divisor fixed for a whole call: division is a shift when it is a power
// of two (the usual block sizes, shard counts and row repeats), else the
// plain division. Only for non-negative dividends.
struct Divisor {
  uint32_t d;
  int32_t log2;  // -1: not a power of two
  __device__ __forceinline__ uint32_t div(uint32_t x) const {
    return log2 >= 0 ? x >> log2 : x / d;
  }
};

inline Divisor make_divisor(int64_t d) {
  Divisor v{static_cast<uint32_t>(d), -1};
  if (d > 0 && (d & (d - 1)) == 0) {
    int l = 0;
    while ((int64_t{1} << l) < d) ++l;
    v.log2 = l;
  }
  return v;
}

struct SelectArgs {
  const void* logits;    // E::T elements
  int64_t ld;            // row stride (elements)
  int64_t shard_stride;  // sharded: elements between shards
  int32_t shards;        // 1 for the unsharded form
  int32_t width;         // unsharded width, or local width of each shard
  const int32_t* row_ks;  // unsharded only, nullable
  const int32_t* row_ke;  // unsharded: window ends; sharded: global ends
  int32_t row_repeat;
  int32_t block_size;    // unsharded block, or local block of each shard
  int32_t global_block_size;
  int32_t nb;            // blocks per output row
  int32_t nb_data;       // blocks that can hold data (sharded: min(ceil(lw/lbs), nbg))
  int32_t pin_newest;    // unsharded only
  int32_t topk;
  int32_t kpad;
  int32_t* out;
  int64_t ld_out;
  void* scores;          // E::T elements, nullable
  int64_t ld_scores;
  int32_t split;        // CTAs per row at most (grid = rows * split)
  int32_t chunk;        // blocks per CTA of a split row (>= nb when split == 1)
  uint32_t* ws_keys;    // split > 1: [rows, nb] block keys
  uint32_t* ws_count;   // split > 1: [rows] arrival counters (zero between calls)
  int64_t rows;         // rows of the call
  int32_t reverse;      // select_warp_kernel: take rows last to first
  int32_t rank_cta;     // select_kernel: the whole CTA ranks every row
  Divisor by_repeat;    // row_repeat
  Divisor by_block;     // block_size
  Divisor by_gblock;    // global_block_size
  Divisor by_shards;    // shards
};

template <typename E>
struct RowPlan {
  const typename E::T* origin;
  int32_t len_max;
  int32_t nblk;       // blocks holding in-window data
  int32_t pin_block;  // -1: none
  int vec, lpb_log2;
  int shift;          // vec == kVecShift: elements past the 16-byte boundary
};

// Adds `units` of a row's `total` to the row's counter and returns true for
// the CTA whose addition completes the total. That CTA writes 0 back, so a
// completed call leaves its counters at zero. A counter word can also hold
// block-key data left by an earlier call of another shape; every block key
// is >= key(-inf) while a count is < total <= 16384 / 32, so such a word is
// read as zero. Each failed CAS but the first means another CTA of the row
// succeeded, so at most `total` + 1 attempts are made.
__device__ __forceinline__ bool arrive_units(uint32_t* counter, uint32_t units, uint32_t total) {
  uint32_t seen = 0u;
  for (uint32_t i = 0; i < total + 2u; ++i) {
    const uint32_t count = (seen >= kKeyNegInf ? 0u : seen) + units;
    const uint32_t prev = atomicCAS(counter, seen, count == total ? 0u : count);
    if (prev == seen) return count == total;
    seen = prev;
  }
  return false;
}

// The streaming plan of one window: n elements starting at column s of a
// row whose element 0 is at `base`; blocks counted from s; no pin. A window
// off the 16-byte grid still reads 16-byte vectors when the block splits
// into a power of two of them and the aligned base stays inside the row
// (s >= shift).
template <typename E>
__device__ __forceinline__ RowPlan<E> plan_window(const typename E::T* base, int32_t s,
                                                  int32_t n, int32_t block_size, Divisor by_block) {
  constexpr int V16 = 16 / E::kBytes;  // elements per 16-byte vector
  RowPlan<E> p;
  p.origin = base + s;
  p.len_max = n;
  p.nblk = static_cast<int32_t>(
      by_block.div(static_cast<uint32_t>(n) + static_cast<uint32_t>(block_size) - 1u));
  p.pin_block = -1;
  p.shift = static_cast<int>((reinterpret_cast<uintptr_t>(p.origin) / E::kBytes) & (V16 - 1));
  const int32_t lpbv = block_size / V16;
  if (p.shift != 0 && s >= p.shift && block_size % V16 == 0 && (lpbv & (lpbv - 1)) == 0) {
    p.vec = kVecShift;
    p.lpb_log2 = __ffs(lpbv) - 1;
  } else {
    p.vec = choose_vec<E>(p.origin, block_size, &p.lpb_log2);
  }
  return p;
}

// Window of an unsharded row: e = min(ke, width), s = min(max(ks, 0), e).
// Every thread computes the same plan from the row's bounds.
template <typename E>
__device__ __forceinline__ RowPlan<E> plan_unsharded(const typename E::T* logits, int64_t ld,
                                                     int32_t width, const int32_t* row_ks,
                                                     const int32_t* row_ke, Divisor by_repeat,
                                                     int32_t block_size, Divisor by_block,
                                                     int32_t pin_newest, int64_t row) {
  const uint32_t g = by_repeat.div(static_cast<uint32_t>(row));
  const int32_t ks = row_ks ? __ldg(row_ks + g) : 0;
  const int32_t ke = __ldg(row_ke + g);
  const int32_t e = min(ke, width);
  const int32_t s = min(max(ks, 0), e);
  const int32_t n = e > s ? e - s : 0;
  RowPlan<E> p = plan_window<E>(logits + row * ld, s, n, block_size, by_block);
  p.pin_block = (pin_newest && n > 0) ? static_cast<int32_t>(by_block.div(n - 1)) : -1;
  return p;
}

// A group of shards that share their window start (and so its alignment),
// streamed 8 shards per slab with the group's plan (16-, 8- or 4-byte
// vectors, or elements), or 4 shards and 2 vectors per lane for shifted
// 16-byte vectors (measured faster than 8 x 1 there, which spills).
template <typename E>
__device__ __forceinline__ void stream_group(const Window<E>& w, const RowPlan<E>& p,
                                             int32_t block_size, int32_t b0, int32_t b1,
                                             uint32_t* keys) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  constexpr int V16 = 16 / E::kBytes, V8 = 8 / E::kBytes, V4 = 4 / E::kBytes;
  if (b0 >= b1) return;
  if (p.vec == kVecShift) {
    ShiftGroups<E> sg;
    sg.base[0] = sg.base[1] = p.origin - p.shift;
    sg.r[0] = sg.r[1] = p.shift;
    sg.split = 0;
    sg.shard_stride = w.shard_stride;
    sg.shards = w.shards;
    sg.len = w.len;
    sg.v_cap = (w.len_max + p.shift) / V16;
    sg.merge = w.merge;
    stream_shift<E, 2, 4>(sg, p.lpb_log2, b0, b1, keys, 0, warp, nwarps);
  } else if (p.vec == V16)
    stream_pow2<E, V16, 1, 8>(w, p.lpb_log2, b0, b1, keys, 0, warp, nwarps);
  else if (p.vec == V8)
    stream_pow2<E, V8, 2, 8>(w, p.lpb_log2, b0, b1, keys, 0, warp, nwarps);
  else if (p.vec == V4 && V4 > 1)
    stream_pow2<E, (V4 > 1 ? V4 : 2), 4, 8>(w, p.lpb_log2, b0, b1, keys, 0, warp, nwarps);
  else if (p.vec == 1)
    stream_pow2<E, 1, 4, 8>(w, p.lpb_log2, b0, b1, keys, 0, warp, nwarps);
  else
    stream_generic<E, 4, 8>(w, block_size, b0, b1, keys, 0, warp, nwarps);
}

// SVEC elements per vector (0: generic path); 8 shards per batch and NV
// vectors per shard, so that each lane has 8 x 16 bytes in flight (8 x 8
// bytes for single bf16 elements, whose loads fill one register each).
template <typename E, int SVEC>
__device__ __forceinline__ void stream_sharded(const Window<E>& w, int lpb_log2,
                                               int32_t block_size, int32_t b0, int32_t b1,
                                               uint32_t* keys) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if constexpr (SVEC > 0) {
    constexpr int NV = 16 / (SVEC * E::kBytes) < 4 ? 16 / (SVEC * E::kBytes) : 4;
    stream_pow2<E, SVEC, NV, 8>(w, lpb_log2, b0, b1, keys, 0, warp, nwarps);
  } else {
    stream_generic<E, 4, 8>(w, block_size, b0, b1, keys, 0, warp, nwarps);
  }
}

// The row's streaming plan (every thread computes the same one from the
// row's bounds); fills the per-shard window lengths (and, with starts, the
// window starts) in shared memory, which other threads may read only after
// the next barrier.
template <typename E, int MODE, int SVEC>
__device__ __forceinline__ RowPlan<E> plan_row(const SelectArgs& a, int64_t row, int32_t* len,
                                               int32_t* start, int32_t& shard_q,
                                               int32_t& shard_rem) {
  using TE = typename E::T;
  const TE* logits = static_cast<const TE*>(a.logits);
  RowPlan<E> plan;
  if constexpr (MODE == kShardedStarts) {
    // Each shard's window [start[d], start[d] + len[d]) and its blocks
    // count from start[d]; the vector width is chosen per shard later.
    // With x = q * shards + r (0 <= r < shards), shard d holds
    // ceil((x - d) / shards) = q + (d < r) of the global tokens below x, so
    // two divisions give every shard's start and end.
    const uint32_t g = a.by_repeat.div(static_cast<uint32_t>(row));
    const int32_t gke = max(__ldg(a.row_ke + g), 0);
    const int32_t gs = min(max(__ldg(a.row_ks + g), 0), gke);
    const int32_t qe = static_cast<int32_t>(a.by_shards.div(static_cast<uint32_t>(gke)));
    const int32_t re = gke - qe * a.shards;
    shard_q = static_cast<int32_t>(a.by_shards.div(static_cast<uint32_t>(gs)));
    shard_rem = gs - shard_q * a.shards;
    auto window = [&](int d, int32_t& st) {
      const int32_t e = min(qe + (d < re ? 1 : 0), a.width);
      st = min(shard_q + (d < shard_rem ? 1 : 0), e);
      return e - st;
    };
    // A shard's window length is constant on the runs of d cut at
    // shard_rem and re, so its largest value is taken at one of d = 0,
    // shard_rem, re and shards - 1.
    int32_t st;
    const int32_t last = a.shards - 1;
    const int32_t len_max = max(max(window(0, st), window(min(shard_rem, last), st)),
                                max(window(min(re, last), st), window(last, st)));
    for (int d = threadIdx.x; d < a.shards; d += blockDim.x) {
      len[d] = window(d, st);
      start[d] = st;
    }
    plan.origin = logits + row * a.ld;
    plan.len_max = len_max;
    plan.nblk = min(static_cast<int32_t>(
                        a.by_block.div(static_cast<uint32_t>(len_max) + a.block_size - 1u)),
                    a.nb_data);
    plan.pin_block = gke > gs ? static_cast<int32_t>(min(
                                    a.by_gblock.div(static_cast<uint32_t>(gke - gs - 1)),
                                    static_cast<uint32_t>(a.nb - 1)))
                              : -1;
    plan.vec = 0;
    plan.lpb_log2 = 0;
  } else if constexpr (MODE == kSharded) {
    // Shard d holds q + (d < r) of the global tokens below gke = q * shards + r.
    const int32_t gke = max(__ldg(a.row_ke + a.by_repeat.div(static_cast<uint32_t>(row))), 0);
    const int32_t qe = static_cast<int32_t>(a.by_shards.div(static_cast<uint32_t>(gke)));
    const int32_t re = gke - qe * a.shards;
    const int32_t n0 = min(qe + (re > 0 ? 1 : 0), a.width);
    plan.origin = logits + row * a.ld;
    plan.len_max = n0;
    plan.nblk = min(static_cast<int32_t>(
                        a.by_block.div(static_cast<uint32_t>(n0) + a.block_size - 1u)),
                    a.nb_data);
    plan.pin_block = gke >= 1 ? static_cast<int32_t>(min(
                                    a.by_gblock.div(static_cast<uint32_t>(gke - 1)),
                                    static_cast<uint32_t>(a.nb - 1)))
                              : -1;
    plan.vec = SVEC;
    plan.lpb_log2 = SVEC ? __ffs(a.block_size / (SVEC ? SVEC : 1)) - 1 : 0;
    for (int d = threadIdx.x; d < a.shards; d += blockDim.x)
      len[d] = min(qe + (d < re ? 1 : 0), a.width);
  } else {
    plan = plan_unsharded<E>(logits, a.ld, a.width, a.row_ks, a.row_ke, a.by_repeat,
                             a.block_size, a.by_block, a.pin_newest, row);
    if (threadIdx.x == 0) len[0] = plan.len_max;
  }

  return plan;
}

// Streams blocks [b0, b1) of `row` into keys[b0, b1) (initialised to
// key(-inf) by the caller before a barrier), the window-end tails included.
// Called by every thread of the CTA; ends with a barrier.
template <typename E, int MODE, int SVEC>
__device__ __forceinline__ void stream_range(const SelectArgs& a, const RowPlan<E>& plan,
                                             int32_t shard_q, int32_t shard_rem, int32_t b0,
                                             int32_t b1, uint32_t* keys, int32_t* len,
                                             int32_t* start) {
  using TE = typename E::T;
  Window<E> w;
  w.origin = plan.origin;
  w.shard_stride = a.shard_stride;
  w.shards = a.shards;
  w.len = len;
  w.len_max = plan.len_max;
  if (b0 < b1) {
    if constexpr (MODE == kShardedStarts) {
      // With gs = q * shards + rg, shards d < rg start at local column
      // q + 1 and the others at q: two groups whose shards share a start.
      // When the shard stride keeps 16-byte alignment, each group streams
      // like the form without starts (all its shards per slab); the second
      // group merges with atomicMax after a barrier. Otherwise every shard
      // row streams on its own.
      const int32_t rg = a.shards > 1 ? shard_rem : 0;
      const bool grouped = (a.shard_stride * E::kBytes) % 16 == 0;
      // One pass over both groups, read from one aligned base
      // (stream_shift_paired), when the block is a power of two of 16-byte
      // vectors and the base stays inside the rows.
      constexpr int V16 = 16 / E::kBytes;
      const int32_t lpbv = a.block_size / V16;
      bool paired = grouped && a.block_size % V16 == 0 && (lpbv & (lpbv - 1)) == 0;
      PairedShift<E> ps;
      if (paired) {
        const int32_t q = min(shard_q, a.width);
        const TE* o = plan.origin + q;
        const int32_t r0 = static_cast<int32_t>((reinterpret_cast<uintptr_t>(o) / E::kBytes) &
                                                (V16 - 1));
        paired = q >= r0;
        ps.base = o - r0;
        ps.r0 = r0;
        ps.split = rg;
        ps.shard_stride = a.shard_stride;
        ps.shards = a.shards;
        ps.len = len;
        ps.merge = false;
        // A bound on every shard's whole vectors (each shard's own limit is
        // applied in the loop).
        ps.v_cap = (plan.len_max + r0 + 1) / V16;
      }
      if (paired)
        stream_shift_paired<E, 8>(ps, __ffs(lpbv) - 1, b0, b1, keys, 0, threadIdx.x >> 5,
                                  blockDim.x >> 5);
      for (int grp = 0; grp < 2 && !paired; ++grp) {
        const int d_lo = grp == 0 ? rg : 0, d_hi = grp == 0 ? a.shards : rg;
        if (d_lo >= d_hi) continue;
        if (grouped) {
          int32_t lmax = 0;
          for (int d = d_lo; d < d_hi; ++d) lmax = max(lmax, len[d]);
          const int32_t st = grp == 0 ? shard_q : shard_q + 1;
          const int32_t st_c = min(st, a.width);
          const RowPlan<E> pg = plan_window<E>(plan.origin + d_lo * a.shard_stride, st_c, lmax,
                                               a.block_size, a.by_block);
          Window<E> wg;
          wg.origin = pg.origin;
          wg.shard_stride = a.shard_stride;
          wg.shards = d_hi - d_lo;
          wg.len = len + d_lo;
          wg.len_max = lmax;
          wg.merge = grp == 1;
          stream_group<E>(wg, pg, a.block_size, b0, min(b1, pg.nblk), keys);
        } else {
          for (int d = d_lo; d < d_hi; ++d) {
            const RowPlan<E> pd = plan_window<E>(plan.origin + d * a.shard_stride, start[d],
                                                 len[d], a.block_size, a.by_block);
            Window<E> wd;
            wd.origin = pd.origin;
            wd.shard_stride = 0;
            wd.shards = 1;
            wd.len = len + d;
            wd.len_max = len[d];
            wd.merge = true;
            stream_row(wd, pd.vec, pd.shift, pd.lpb_log2, a.block_size, b0,
                       min(b1, pd.nblk), keys, 0, threadIdx.x >> 5, blockDim.x >> 5);
          }
        }
        if (grp == 0) __syncthreads();
      }
    } else if constexpr (MODE == kSharded) {
      stream_sharded<E, SVEC>(w, plan.lpb_log2, a.block_size, b0, b1, keys);
    } else {
      stream_row(w, plan.vec, plan.shift, plan.lpb_log2, a.block_size, b0, b1, keys, 0,
                 threadIdx.x >> 5, blockDim.x >> 5);
    }
  }
  __syncthreads();
  if constexpr (MODE == kShardedStarts) {
    // Shard d's tail on lane d / warps of warp d % warps: every warp takes a
    // share, so the barrier below waits on less.
    const int nwarps = blockDim.x >> 5;
    for (int d = (threadIdx.x & 31) * nwarps + (threadIdx.x >> 5); d < a.shards;
         d += 32 * nwarps) {
      const RowPlan<E> pd = plan_window<E>(plan.origin + d * a.shard_stride, start[d], len[d],
                                           a.block_size, a.by_block);
      Window<E> wd;
      wd.origin = pd.origin;
      wd.shard_stride = 0;
      wd.shards = 1;
      wd.len = len + d;
      wd.len_max = len[d];
      finish_row(wd, pd.vec, pd.shift, a.block_size, b0, min(b1, pd.nblk), keys, 0);
    }
  } else if constexpr (MODE == kSharded) {
    if constexpr (SVEC > 1)
      for (int d = threadIdx.x; d < a.shards; d += blockDim.x)
        commit_partial(load_partial<E, SVEC>(plan.origin + d * a.shard_stride, len[d],
                                             a.block_size, b0, b1),
                       keys, 0);
  } else {
    if (threadIdx.x == 0) finish_row(w, plan.vec, plan.shift, a.block_size, b0, b1, keys, 0);
  }
  __syncthreads();

}

// Pins, ranks and stores one row whose block keys [0, nblk) are final in
// shared memory. Called by every thread of the CTA. Rows of up to 1024 live
// blocks with k <= 32 are ranked by warp 0 alone (topk_warp_wide): the
// other warps leave, and the ranking costs a quarter of the instructions of
// the CTA-wide topk_store.
// Keys [nblk, pin] were set to key(-inf) with the CTA's own blocks; the pin
// becomes +inf inside the ranking. `merged`: the keys were just read back
// from the workspace (a split row), so a barrier comes first.
template <typename E>
__device__ __forceinline__ void rank_row(const SelectArgs& a, int64_t row, int32_t nblk,
                                         int32_t pin_block, uint32_t* keys, uint64_t* cand,
                                         TopkShared& tsh, bool merged) {
  using TE = typename E::T;
  const int32_t n_live = max(nblk, pin_block + 1);
  const int32_t k = min(a.topk, a.nb);
  int32_t* out = a.topk > 0 ? a.out + row * a.ld_out : nullptr;
  TE* scores = a.scores ? static_cast<TE*>(a.scores) + row * a.ld_scores : nullptr;
  if (merged) __syncthreads();
  if (!a.rank_cta && k <= 32 && n_live <= 1024) {
    if (threadIdx.x < 32)
      topk_warp_wide(keys, a.nb, n_live, k, pin_block, cand, max(a.kpad, kRankMax), out, a.topk,
                     scores);
    return;
  }
  topk_store(keys, a.nb, n_live, k, pin_block, cand, a.kpad, out, a.topk, scores, tsh);
}

// Publishes keys [b0, b1) of `row` to the workspace and counts `units` of the
// row's `total` in; returns (to every thread) whether this CTA was the last
// to arrive, in which case keys [0, nblk) now hold the whole row.
__device__ __forceinline__ bool merge_shares(const SelectArgs& a, int64_t row, int32_t nblk,
                                             int32_t b0, int32_t b1, uint32_t units,
                                             uint32_t total, uint32_t* keys, int* s_last) {
  uint32_t* wrow = a.ws_keys + row * a.nb;
  for (int32_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) __stcg(wrow + b, keys[b]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_last = arrive_units(a.ws_count + row, units, total);
  __syncthreads();
  if (!*s_last) return false;
  __threadfence();
  for (int32_t b = threadIdx.x; b < nblk; b += blockDim.x)
    if (b < b0 || b >= b1) keys[b] = __ldcg(wrow + b);
  return true;
}

// Up to `a.split` CTAs per row. A row's in-window blocks are cut from its
// start into parts of `a.chunk` blocks, and CTA i takes part i / rows of row
// i % rows (chunk-major): a short row uses only the parts its data reaches,
// and the CTAs launched last hold the far parts of the longest rows.
// MODE kUnsharded: unsharded rows, vector width chosen per row.
// MODE kSharded: DCP rows; SVEC is the vector width fixed by the host
// (0 = generic path). T: threads per CTA.
template <typename E, int MODE, int SVEC, int T>
__global__ void __launch_bounds__(T, 1024 / T) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw);  // [max(kpad, kRankMax)]
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + max(a.kpad, kRankMax));  // [nb]
  int32_t* len = reinterpret_cast<int32_t*>(keys + ((a.nb + 3) & ~3));   // [shards]
  int32_t* start = len + a.shards;  // [shards], kShardedStarts only
  __shared__ TopkShared tsh;
  __shared__ int s_last;

  const uint32_t rows = static_cast<uint32_t>(a.rows);
  const int64_t row = a.split == 1 ? blockIdx.x : blockIdx.x % rows;
  const int32_t part = a.split == 1 ? 0 : static_cast<int32_t>(blockIdx.x / rows);

  int32_t shard_q = 0, shard_rem = 0;  // kShardedStarts: gs = shard_q * shards + shard_rem
  const RowPlan<E> plan = plan_row<E, MODE, SVEC>(a, row, len, start, shard_q, shard_rem);
  const int32_t nblk = plan.nblk;
  const int32_t parts = max(1, (nblk + a.chunk - 1) / a.chunk);
  if (part >= parts) return;  // past the row's data
  const int32_t b0 = part * a.chunk;
  const int32_t b1 = min(b0 + a.chunk, nblk);

  // This CTA's blocks, and the blocks past the data up to the pin (which can
  // lie past the data in the DCP form; no stream writes them), start at
  // key(-inf).
  for (int32_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) keys[b] = kKeyNegInf;
  for (int32_t b = nblk + threadIdx.x; b <= plan.pin_block; b += blockDim.x) keys[b] = kKeyNegInf;
  __syncthreads();
  stream_range<E, MODE, SVEC>(a, plan, shard_q, shard_rem, b0, b1, keys, len, start);
  // Publish this share, count in; only the last CTA of the row goes on.
  if (parts > 1 &&
      !merge_shares(a, row, nblk, b0, b1, 1u, static_cast<uint32_t>(parts), keys, &s_last))
    return;
  rank_row<E>(a, row, nblk, plan.pin_block, keys, cand, tsh, parts > 1);
}

// Shared memory per warp in select_warp_kernel: candidates, keys, length.
__host__ __device__ __forceinline__ size_t warp_slice_bytes(int32_t nb) {
  return static_cast<size_t>(kWarpCand) * 8 + static_cast<size_t>((nb + 3) & ~3) * 4 + 16;
}

// One row per warp, W warps per CTA, for short unsharded rows: each warp
// streams its row alone (stream_row with one warp) into its own key array
// and ranks it with topk_warp; no CTA barrier anywhere, so W rows of a CTA
// proceed independently and up to 32 rows are in flight per SM.
template <typename E, int W>
__global__ void __launch_bounds__(W * 32, 1024 / (W * 32)) select_warp_kernel(const SelectArgs a) {
  using TE = typename E::T;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Rows are taken last to first: in a causally ordered chunk (packed
  // prefill) later rows are longer, so the longest rows start first and the
  // launch ends on short ones.
  const int64_t slot = static_cast<int64_t>(blockIdx.x) * W + warp;
  if (slot >= a.rows) return;
  const int64_t row = a.reverse ? a.rows - 1 - slot : slot;
  unsigned char* slice = smem_raw + warp * warp_slice_bytes(a.nb);
  uint64_t* cand = reinterpret_cast<uint64_t*>(slice);
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + kWarpCand);
  int32_t* len = reinterpret_cast<int32_t*>(keys + ((a.nb + 3) & ~3));

  const RowPlan<E> plan =
      plan_unsharded<E>(static_cast<const TE*>(a.logits), a.ld, a.width, a.row_ks, a.row_ke,
                        a.by_repeat, a.block_size, a.by_block, a.pin_newest, row);
  if (lane == 0) len[0] = plan.len_max;
  const int32_t nblk = plan.nblk;
  for (int32_t b = lane; b < nblk; b += 32) keys[b] = kKeyNegInf;
  __syncwarp();
  Window<E> w;
  w.origin = plan.origin;
  w.shard_stride = 0;
  w.shards = 1;
  w.len = len;
  w.len_max = plan.len_max;
  if (nblk > 0)
    stream_row(w, plan.vec, plan.shift, plan.lpb_log2, a.block_size, 0, nblk, keys, 0, 0, 1);
  __syncwarp();
  if (lane == 0) finish_row(w, plan.vec, plan.shift, a.block_size, 0, nblk, keys, 0);
  __syncwarp();
  topk_warp(keys, a.nb, nblk, min(a.topk, a.nb), plan.pin_block, cand,
            a.topk > 0 ? a.out + row * a.ld_out : nullptr, a.topk,
            a.scores ? static_cast<TE*>(a.scores) + row * a.ld_scores : nullptr);
}

struct ScoresArgs {
  const void* logits;  // E::T elements
  int64_t ld;
  int32_t width;
  const int32_t* row_ks;
  const int32_t* row_ke;
  int32_t row_repeat;
  int32_t block_size;
  int32_t nb;
  int32_t pin_newest;
  int32_t chunk;   // blocks per CTA
  int32_t chunks;  // CTAs per row
  void* scores;        // E::T elements
  int64_t ld_scores;
  Divisor by_repeat;
  Divisor by_block;
};

template <typename E>
__global__ void __launch_bounds__(kThreads, 4) block_scores_kernel(const ScoresArgs a) {
  using TE = typename E::T;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);  // [chunk]
  __shared__ int32_t len[1];
  const int64_t row = blockIdx.x / a.chunks;
  const int32_t c0 = static_cast<int32_t>(blockIdx.x % a.chunks) * a.chunk;
  const int32_t c1 = min(c0 + a.chunk, a.nb);

  const RowPlan<E> plan =
      plan_unsharded<E>(static_cast<const TE*>(a.logits), a.ld, a.width, a.row_ks, a.row_ke,
                        a.by_repeat, a.block_size, a.by_block, a.pin_newest, row);
  if (threadIdx.x == 0) len[0] = plan.len_max;
  for (int32_t b = threadIdx.x; b < c1 - c0; b += blockDim.x) keys[b] = kKeyNegInf;
  __syncthreads();
  const int32_t b0 = min(c0, plan.nblk), b1 = min(c1, plan.nblk);
  Window<E> w;
  w.origin = plan.origin;
  w.shard_stride = 0;
  w.shards = 1;
  w.len = len;
  w.len_max = plan.len_max;
  if (b0 < b1)
    stream_row(w, plan.vec, plan.shift, plan.lpb_log2, a.block_size, b0, b1, keys, c0,
               threadIdx.x >> 5, blockDim.x >> 5);
  __syncthreads();
  if (threadIdx.x == 0) finish_row(w, plan.vec, plan.shift, a.block_size, b0, b1, keys, c0);
  __syncthreads();
  if (threadIdx.x == 0 && plan.pin_block >= c0 && plan.pin_block < c1)
    keys[plan.pin_block - c0] = kKeyPosInf;
  __syncthreads();
  TE* srow = static_cast<TE*>(a.scores) + row * a.ld_scores;
  for (int32_t b = c0 + threadIdx.x; b < c1; b += blockDim.x) put_score(srow + b, keys[b - c0]);
}

__global__ void fill_minus_one_kernel(int32_t* out, int64_t rows, int32_t cols, int64_t ld) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x)
    out[(i / cols) * ld + (i % cols)] = -1;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Launch-shape overrides (dsa_select_set_launch_override): 0 leaves the
// choice to the launcher. Set explicitly by tests and tuning sweeps; nothing
// in the library reads them from the process settings.
std::atomic<int> g_split_override{0};    // CTAs per row with a workspace, 1..8
std::atomic<int> g_threads_override{0};  // 128 or 256 threads per CTA
std::atomic<int> g_warp_off{0};          // 1: never one row per warp
std::atomic<int> g_warp_in_order{0};     // 1: one row per warp, rows in order
std::atomic<int> g_rank_cta{0};          // select_kernel ranking: 1 whole CTA, 2 one warp

int32_t next_pow2(int32_t x) {
  int32_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Workspace layout (select_pipe.h): a 256-byte header (the pipelined
// kernels' unit queue), rows arrival counters (uint32), then rows * nb block
// keys (uint32), each part 256-byte aligned.
size_t workspace_bytes(int64_t rows, int64_t nb) { return ws_total_bytes(rows, nb); }

// Streaming multiprocessors of the current device, cached per device.
int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launch shape (measured on GB300 over the workloads):
//  - 128 threads per CTA (8 CTAs per SM at 64 registers): a CTA's top-k
//    leaves fewer threads idle and more rows are in flight. (256 threads
//    measured slower for the 512 KiB rows of the long workload, 82.6 us
//    against 78.9 us with 4 CTAs per row.)
//  - Rows are split over S CTAs (with a workspace) only while there are fewer
//    than ~3 waves of CTAs, and never below 64 KiB per CTA: small CTA shares
//    are latency-bound, and a full machine gains nothing from splitting.
struct Shape {
  int split;
  int threads;
};

Shape choose_shape(int64_t max_row_bytes, int64_t rows, bool have_workspace) {
  Shape sh{1, 128};
  if (const int t = g_threads_override.load(std::memory_order_relaxed)) sh.threads = t;
  if (have_workspace) {
    const int64_t slots = static_cast<int64_t>(sm_count()) * (1024 / sh.threads);
    int split = 1;
    while (split < kMaxSplit && rows * split < 3 * slots &&
           max_row_bytes / (2 * split) >= 64 * 1024)
      split <<= 1;
    const int forced = g_split_override.load(std::memory_order_relaxed);
    sh.split = forced ? forced : split;
  }
  return sh;
}

// Opts a kernel in to `smem` bytes of dynamic shared memory on the current
// device (static plus dynamic shared memory above 48 KiB needs the opt-in).
// Remembers the largest size set per (kernel, device) so repeated launches
// make no runtime call.
struct SmemOptIn {
  const void* fn;
  int device;
  size_t bytes;
};
std::mutex g_smem_mu;
SmemOptIn g_smem_table[64];
int g_smem_used = 0;

template <typename K>
cudaError_t set_smem_attr(K kernel, size_t smem) {
  if (smem == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const void* fn = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (int i = 0; i < g_smem_used; ++i) {
    if (g_smem_table[i].fn == fn && g_smem_table[i].device == dev) {
      if (g_smem_table[i].bytes >= smem) return cudaSuccess;
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err == cudaSuccess) g_smem_table[i].bytes = smem;
      return err;
    }
  }
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err == cudaSuccess && g_smem_used < 64) g_smem_table[g_smem_used++] = {fn, dev, smem};
  return err;
}

template <typename K>
dsa_status launch_select(K kernel, const SelectArgs& a, int64_t rows, int threads, size_t smem,
                         cudaStream_t stream) {
  if (set_smem_attr(kernel, smem) != cudaSuccess) return DSA_ECUDA;
  kernel<<<static_cast<unsigned>(rows * a.split), threads, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

// Instantiates the kernel for the chosen thread count.
template <typename E, int MODE, int SVEC>
dsa_status launch_shape(const SelectArgs& a, int64_t rows, const Shape& sh, size_t smem,
                        cudaStream_t stream) {
  if (sh.threads == 128)
    return launch_select(select_kernel<E, MODE, SVEC, 128>, a, rows, 128, smem, stream);
  return launch_select(select_kernel<E, MODE, SVEC, 256>, a, rows, 256, smem, stream);
}

// Fills the workspace fields of `a` for the chosen shape.
void attach_workspace(SelectArgs& a, int64_t rows, void* workspace, const Shape& sh) {
  a.split = sh.split;
  a.rows = rows;
  // The part size of an even split of the longest row, in whole units.
  const int32_t units = (a.nb_data + kSplitUnit - 1) / kSplitUnit;
  a.chunk = sh.split > 1 ? std::max(1, (units + sh.split - 1) / sh.split) * kSplitUnit
                         : std::max(a.nb, 1);
  if (sh.split == 1) return;
  a.ws_count = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws_counts_offset());
  a.ws_keys = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws_keys_offset(rows));
}

dsa_status fill_minus_one(int32_t* out, int64_t rows, int32_t cols, int64_t ld, cudaStream_t s) {
  if (rows == 0 || cols == 0) return DSA_OK;
  const int64_t total = rows * cols;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, 4096));
  fill_minus_one_kernel<<<grid, 256, 0, s>>>(out, rows, cols, ld);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

// Dynamic shared memory of select_kernel: candidates, block keys (padded to
// a multiple of 4 for 16-byte loads), and the shard lengths and starts.
size_t select_smem(int32_t kpad, int32_t nb, int32_t shards) {
  return static_cast<size_t>(std::max(kpad, kRankMax)) * 8 +
         static_cast<size_t>((nb + 3) & ~3) * 4 + static_cast<size_t>(shards) * 8;
}


}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_EINVAL: return "invalid argument";
    case DSA_ECUDA: return "CUDA runtime or launch failure";
    case DSA_EUNSUPPORTED: return "beyond this build's limits";
    default: return "unknown status";
  }
}

int32_t dsa_select_max_blocks(void) { return kMaxSelectBlocks; }
int32_t dsa_select_max_shards(void) { return kMaxShards; }

size_t dsa_select_workspace_bytes(int64_t rows, int64_t nblocks) {
  if (rows < 0 || nblocks < 0) return 0;
  return workspace_bytes(rows, nblocks);
}

dsa_status dsa_select_set_launch_override(int32_t knob, int32_t value) {
  switch (knob) {
    case DSA_LAUNCH_SPLIT:
      if (value < 0 || value > kMaxSplit) return DSA_EINVAL;
      g_split_override.store(value);
      return DSA_OK;
    case DSA_LAUNCH_THREADS:
      if (value != 0 && value != 128 && value != 256) return DSA_EINVAL;
      g_threads_override.store(value);
      return DSA_OK;
    case DSA_LAUNCH_WARP_ROWS:
      if (value < 0 || value > 1) return DSA_EINVAL;
      g_warp_off.store(value);
      return DSA_OK;
    case DSA_LAUNCH_WARP_ORDER:
      if (value < 0 || value > 1) return DSA_EINVAL;
      g_warp_in_order.store(value);
      return DSA_OK;
    case DSA_LAUNCH_PIPELINE:
      if (value < 0 || value > 3) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_SPLIT:
      if (value < 0 || value > 8) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_STAGES:
      if (value != 0 && (value < 2 || value > 16)) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_STAGE_KB:
      if (value != 0 && (value < 4 || value > 64)) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_SCHED:
      if (value < 0 || value > 1) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_WARPS:
      if (value != 0 && value != 4 && value != 8) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_CTAS:
      if (value < 0 || value > 4) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_STAGE_OWNER:
      if (value < 0 || value > 1) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_PIPE_ORDER:
      if (value < 0 || value > 3) return DSA_EINVAL;
      pipe_set_override(knob, value);
      return DSA_OK;
    case DSA_LAUNCH_RANK_CTA:
      if (value < 0 || value > 2) return DSA_EINVAL;
      g_rank_cta.store(value);
      pipe_set_override(knob, value);
      return DSA_OK;
    default:
      return DSA_EINVAL;
  }
}

}  // extern "C"

namespace dsa {
namespace {

template <typename E>
dsa_status block_scores_impl(const typename E::T* logits, int64_t rows, int64_t width,
                             int64_t ld_logits, const int32_t* row_ks, const int32_t* row_ke,
                             int32_t block_size, int32_t row_repeat, int32_t pin_newest,
                             typename E::T* scores_out, int64_t ld_scores, void* stream) {
  if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1) return DSA_EINVAL;
  if (rows == 0 || width == 0) return DSA_OK;
  if (!logits || !row_ke || !scores_out || ld_logits < width) return DSA_EINVAL;
  const int64_t nb = (width + block_size - 1) / block_size;
  if (ld_scores < nb) return DSA_EINVAL;
  if (width > INT32_MAX - 64) return DSA_EUNSUPPORTED;

  ScoresArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.width = static_cast<int32_t>(width);
  a.row_ks = row_ks;
  a.row_ke = row_ke;
  a.row_repeat = row_repeat;
  a.block_size = block_size;
  a.by_repeat = make_divisor(row_repeat);
  a.by_block = make_divisor(block_size);
  a.nb = static_cast<int32_t>(nb);
  a.pin_newest = pin_newest != 0;
  // About 64 KiB of logits per CTA, at least 32 blocks, at most 4096.
  int64_t chunk = (64 * 1024 / E::kBytes) / block_size;
  chunk = std::max<int64_t>(32, std::min<int64_t>(4096, chunk));
  chunk = std::min<int64_t>(chunk, nb);
  a.chunk = static_cast<int32_t>(chunk);
  a.chunks = static_cast<int32_t>((nb + chunk - 1) / chunk);
  a.scores = scores_out;
  a.ld_scores = ld_scores;
  const size_t smem = static_cast<size_t>(chunk) * 4;
  if (set_smem_attr(block_scores_kernel<E>, smem) != cudaSuccess) return DSA_ECUDA;
  const int64_t grid = rows * a.chunks;
  if (grid > INT32_MAX) return DSA_EUNSUPPORTED;
  block_scores_kernel<E><<<static_cast<unsigned>(grid), kThreads, smem,
                           static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

template <typename E>
dsa_status select_impl(const typename E::T* logits, int64_t rows, int64_t width,
                       int64_t ld_logits, const int32_t* row_ks, const int32_t* row_ke,
                       int32_t topk_blocks, int32_t block_size, int32_t row_repeat,
                       int32_t pin_newest, int32_t* out, int64_t ld_out,
                       typename E::T* scores_out, int64_t ld_scores, void* workspace,
                       size_t workspace_size, void* stream) {
  if (rows < 0 || width < 0 || topk_blocks < 0 || block_size < 1 || row_repeat < 1)
    return DSA_EINVAL;
  if (rows == 0) return DSA_OK;
  if (topk_blocks > 0 && (!out || ld_out < topk_blocks)) return DSA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (width == 0) return fill_minus_one(out, rows, topk_blocks, ld_out, s);
  if (!logits || !row_ke || ld_logits < width) return DSA_EINVAL;
  const int64_t nb = (width + block_size - 1) / block_size;
  if (scores_out && ld_scores < nb) return DSA_EINVAL;
  if (topk_blocks == 0 && !scores_out) return DSA_OK;
  if (nb > kMaxSelectBlocks || width > INT32_MAX - 8192) return DSA_EUNSUPPORTED;
  if (rows > INT32_MAX / kMaxSplit) return DSA_EUNSUPPORTED;

  SelectArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = 0;
  a.shards = 1;
  a.width = static_cast<int32_t>(width);
  a.row_ks = row_ks;
  a.row_ke = row_ke;
  a.row_repeat = row_repeat;
  a.block_size = block_size;
  a.by_repeat = make_divisor(row_repeat);
  a.by_block = make_divisor(block_size);
  a.nb = static_cast<int32_t>(nb);
  a.nb_data = a.nb;
  a.pin_newest = pin_newest != 0;
  a.topk = topk_blocks;
  a.kpad = next_pow2(std::max<int32_t>(1, std::min<int32_t>(topk_blocks, a.nb)));
  a.rank_cta = g_rank_cta.load(std::memory_order_relaxed) == 1;
  a.out = out;
  a.ld_out = ld_out;
  a.scores = scores_out;
  a.ld_scores = ld_scores;
  const int64_t row_bytes = width * E::kBytes;
  {
    PipeCall pc{};
    pc.elem_bytes = E::kBytes;
    pc.mode = kPipeUnsharded;
    pc.logits = logits;
    pc.ld = ld_logits;
    pc.shard_stride = 0;
    pc.shards = 1;
    pc.width = a.width;
    pc.row_ks = row_ks;
    pc.row_ke = row_ke;
    pc.row_repeat = row_repeat;
    pc.block_size = block_size;
    pc.global_block_size = block_size;
    pc.nb = a.nb;
    pc.nb_data = a.nb;
    pc.pin_newest = a.pin_newest;
    pc.topk = topk_blocks;
    pc.out = out;
    pc.ld_out = ld_out;
    pc.scores = scores_out;
    pc.ld_scores = ld_scores;
    pc.rows = rows;
    pc.workspace = workspace;
    pc.workspace_size = workspace_size;
    if (pipe_takes(pc)) {
      const dsa_status st = pipe_select(pc, stream);
      if (st != kPipeDeclined) return st;
    }
  }
  // Many short rows: one row per warp (32 rows in flight per SM instead of
  // 8). With few rows a CTA per row keeps more of the GPU busy.
  if (!g_warp_off.load(std::memory_order_relaxed) && row_bytes <= 64 * 1024 &&
      topk_blocks <= 32 && a.nb <= 2048 && rows >= 8 * static_cast<int64_t>(sm_count())) {
    constexpr int W = 4;
    a.split = 1;
    a.rows = rows;
    a.reverse = !g_warp_in_order.load(std::memory_order_relaxed);
    const size_t smem = W * warp_slice_bytes(a.nb);
    if (set_smem_attr(select_warp_kernel<E, W>, smem) != cudaSuccess) return DSA_ECUDA;
    select_warp_kernel<E, W><<<static_cast<unsigned>((rows + W - 1) / W), W * 32, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
  }
  const bool ws = workspace && workspace_size >= workspace_bytes(rows, a.nb);
  const size_t smem = select_smem(a.kpad, a.nb, 1);
  const Shape sh = choose_shape(row_bytes, rows, ws);
  attach_workspace(a, rows, workspace, sh);
  return launch_shape<E, kUnsharded, 0>(a, rows, sh, smem, s);
}

// Argument checks of the sharded selection, done on the host before anything
// is enqueued: a status < 0 is the call's error, kNoWork means DSA_OK with
// nothing to do, DSA_OK means go on.
constexpr int kNoWork = 1;

int sharded_precheck(const void* logits, int32_t shards, int64_t rows, int64_t local_width,
                     int64_t ld_logits, int64_t shard_stride, const int32_t* global_row_ke,
                     int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
                     int32_t topk_blocks, const int32_t* out, int64_t ld_out,
                     const void* scores_out, int64_t ld_scores) {
  if (shards < 1 || rows < 0 || local_width < 0 || topk_blocks < 0 || global_block_size < 1 ||
      global_block_size % shards != 0 || row_repeat < 1 || ld_logits < local_width ||
      shard_stride < 0)
    return DSA_EINVAL;
  if (rows == 0) return kNoWork;
  if (!global_row_ke || (topk_blocks > 0 && (!out || ld_out < topk_blocks))) return DSA_EINVAL;
  if (local_width > 0 && !logits) return DSA_EINVAL;
  const int32_t nbg = std::max<int32_t>(max_global_blocks, 1);
  if (scores_out && ld_scores < nbg) return DSA_EINVAL;
  if (topk_blocks == 0 && !scores_out) return kNoWork;
  if (nbg > kMaxSelectBlocks || shards > kMaxShards || local_width > INT32_MAX - 8192)
    return DSA_EUNSUPPORTED;
  if (rows > INT32_MAX / kMaxSplit) return DSA_EUNSUPPORTED;
  return DSA_OK;
}

template <typename E>
dsa_status select_sharded_impl(const typename E::T* logits, int32_t shards, int64_t rows,
                               int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                               const int32_t* global_row_ks, const int32_t* global_row_ke,
                               int32_t global_block_size,
                               int32_t max_global_blocks, int32_t row_repeat,
                               int32_t topk_blocks, int32_t* out, int64_t ld_out,
                               typename E::T* scores_out, int64_t ld_scores, void* workspace,
                               size_t workspace_size, void* stream) {
  const int pre = sharded_precheck(logits, shards, rows, local_width, ld_logits, shard_stride,
                                   global_row_ke, global_block_size, max_global_blocks,
                                   row_repeat, topk_blocks, out, ld_out, scores_out, ld_scores);
  if (pre < 0) return static_cast<dsa_status>(pre);
  if (pre == kNoWork) return DSA_OK;
  const int32_t nbg = std::max<int32_t>(max_global_blocks, 1);

  const int32_t lbs = global_block_size / shards;
  SelectArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = shard_stride;
  a.shards = shards;
  a.width = static_cast<int32_t>(local_width);
  a.row_ks = global_row_ks;
  a.row_ke = global_row_ke;
  a.row_repeat = row_repeat;
  a.block_size = lbs;
  a.global_block_size = global_block_size;
  a.by_repeat = make_divisor(row_repeat);
  a.by_block = make_divisor(lbs);
  a.by_gblock = make_divisor(global_block_size);
  a.by_shards = make_divisor(shards);
  a.nb = nbg;
  a.nb_data = static_cast<int32_t>(std::min<int64_t>((local_width + lbs - 1) / lbs, nbg));
  a.pin_newest = 0;
  a.topk = topk_blocks;
  a.kpad = next_pow2(std::max<int32_t>(1, std::min<int32_t>(topk_blocks, nbg)));
  // The fp32 DCP form without starts streams at about 0.91 of the copy
  // bandwidth: there the whole CTA ranks, which frees the CTA's slot sooner
  // (86.0 against 86.7 us on the [8, 4096, 8192] workload). The other forms
  // are issue-bound and rank with one warp.
  {
    const int rc = g_rank_cta.load(std::memory_order_relaxed);
    a.rank_cta = rc == 1 || (rc == 0 && !global_row_ks && sizeof(typename E::T) == 4);
  }
  a.out = out;
  a.ld_out = ld_out;
  a.scores = scores_out;
  a.ld_scores = ld_scores;

  // One vector width (in elements) for every shard row: all shard origins
  // must share the alignment and the local block must split into a power of
  // two of vectors.
  auto pow2 = [](int32_t x) { return x > 0 && (x & (x - 1)) == 0; };
  const uintptr_t base = reinterpret_cast<uintptr_t>(logits);
  auto aligned = [&](int vec) {
    return lbs % vec == 0 && pow2(lbs / vec) && (base % (E::kBytes * vec)) == 0 &&
           ld_logits % vec == 0 && shard_stride % vec == 0;
  };
  {
    PipeCall pc{};
    pc.elem_bytes = E::kBytes;
    pc.mode = global_row_ks ? kPipeShardedStarts : kPipeSharded;
    pc.logits = logits;
    pc.ld = ld_logits;
    pc.shard_stride = shard_stride;
    pc.shards = shards;
    pc.width = a.width;
    pc.row_ks = global_row_ks;
    pc.row_ke = global_row_ke;
    pc.row_repeat = row_repeat;
    pc.block_size = lbs;
    pc.global_block_size = global_block_size;
    pc.nb = a.nb;
    pc.nb_data = a.nb_data;
    pc.pin_newest = 0;
    pc.topk = topk_blocks;
    pc.out = out;
    pc.ld_out = ld_out;
    pc.scores = scores_out;
    pc.ld_scores = ld_scores;
    pc.rows = rows;
    pc.workspace = workspace;
    pc.workspace_size = workspace_size;
    if (local_width > 0 && pipe_takes(pc)) {
      const dsa_status st = pipe_select(pc, stream);
      if (st != kPipeDeclined) return st;
    }
  }
  const size_t smem = select_smem(a.kpad, a.nb, shards);
  const bool ws = workspace && workspace_size >= workspace_bytes(rows, a.nb);
  const Shape sh = choose_shape(local_width * E::kBytes * shards, rows, ws);
  attach_workspace(a, rows, workspace, sh);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // With starts every shard row is planned on its own in the kernel.
  if (global_row_ks) return launch_shape<E, kShardedStarts, 0>(a, rows, sh, smem, s);
  constexpr int V16 = 16 / E::kBytes, V8 = 8 / E::kBytes, V4 = 4 / E::kBytes;
  if (aligned(V16)) return launch_shape<E, kSharded, V16>(a, rows, sh, smem, s);
  if (aligned(V8)) return launch_shape<E, kSharded, V8>(a, rows, sh, smem, s);
  if constexpr (V4 > 1) {
    if (aligned(V4)) return launch_shape<E, kSharded, V4>(a, rows, sh, smem, s);
  }
  if (pow2(lbs)) return launch_shape<E, kSharded, 1>(a, rows, sh, smem, s);
  return launch_shape<E, kSharded, 0>(a, rows, sh, smem, s);
}

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status dsa_block_scores(const float* logits, int64_t rows, int64_t width, int64_t ld_logits,
                            const int32_t* row_ks, const int32_t* row_ke, int32_t block_size,
                            int32_t row_repeat, int32_t pin_newest, float* scores_out,
                            int64_t ld_scores, void* stream) {
  return block_scores_impl<F32>(logits, rows, width, ld_logits, row_ks, row_ke, block_size,
                                row_repeat, pin_newest, scores_out, ld_scores, stream);
}

dsa_status dsa_block_scores_bf16(const uint16_t* logits, int64_t rows, int64_t width,
                                 int64_t ld_logits, const int32_t* row_ks, const int32_t* row_ke,
                                 int32_t block_size, int32_t row_repeat, int32_t pin_newest,
                                 uint16_t* scores_out, int64_t ld_scores, void* stream) {
  return block_scores_impl<BF16>(logits, rows, width, ld_logits, row_ks, row_ke, block_size,
                                 row_repeat, pin_newest, scores_out, ld_scores, stream);
}

dsa_status dsa_select_candidate_blocks(const float* logits, int64_t rows, int64_t width,
                                       int64_t ld_logits, const int32_t* row_ks,
                                       const int32_t* row_ke, int32_t topk_blocks,
                                       int32_t block_size, int32_t row_repeat,
                                       int32_t pin_newest, int32_t* out, int64_t ld_out,
                                       float* scores_out, int64_t ld_scores, void* workspace,
                                       size_t workspace_size, void* stream) {
  return select_impl<F32>(logits, rows, width, ld_logits, row_ks, row_ke, topk_blocks,
                          block_size, row_repeat, pin_newest, out, ld_out, scores_out, ld_scores,
                          workspace, workspace_size, stream);
}

dsa_status dsa_select_candidate_blocks_bf16(const uint16_t* logits, int64_t rows, int64_t width,
                                            int64_t ld_logits, const int32_t* row_ks,
                                            const int32_t* row_ke, int32_t topk_blocks,
                                            int32_t block_size, int32_t row_repeat,
                                            int32_t pin_newest, int32_t* out, int64_t ld_out,
                                            uint16_t* scores_out, int64_t ld_scores,
                                            void* workspace, size_t workspace_size,
                                            void* stream) {
  return select_impl<BF16>(logits, rows, width, ld_logits, row_ks, row_ke, topk_blocks,
                           block_size, row_repeat, pin_newest, out, ld_out, scores_out,
                           ld_scores, workspace, workspace_size, stream);
}

dsa_status dsa_select_candidate_blocks_sharded(const float* logits, int32_t shards, int64_t rows,
                                               int64_t local_width, int64_t ld_logits,
                                               int64_t shard_stride,
                                               const int32_t* global_row_ke,
                                               int32_t global_block_size,
                                               int32_t max_global_blocks, int32_t row_repeat,
                                               int32_t topk_blocks, int32_t* out, int64_t ld_out,
                                               float* scores_out, int64_t ld_scores,
                                               void* workspace, size_t workspace_size,
                                               void* stream) {
  return select_sharded_impl<F32>(logits, shards, rows, local_width, ld_logits, shard_stride,
                                  nullptr, global_row_ke, global_block_size, max_global_blocks,
                                  row_repeat, topk_blocks, out, ld_out, scores_out, ld_scores,
                                  workspace, workspace_size, stream);
}

dsa_status dsa_select_candidate_blocks_sharded_bf16(
    const uint16_t* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ke, int32_t global_block_size,
    int32_t max_global_blocks, int32_t row_repeat, int32_t topk_blocks, int32_t* out,
    int64_t ld_out, uint16_t* scores_out, int64_t ld_scores, void* workspace,
    size_t workspace_size, void* stream) {
  return select_sharded_impl<BF16>(logits, shards, rows, local_width, ld_logits, shard_stride,
                                   nullptr, global_row_ke, global_block_size, max_global_blocks,
                                   row_repeat, topk_blocks, out, ld_out, scores_out, ld_scores,
                                   workspace, workspace_size, stream);
}

dsa_status dsa_select_candidate_blocks_sharded_starts(
    const float* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ks, const int32_t* global_row_ke,
    int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
    int32_t topk_blocks, int32_t* out, int64_t ld_out, float* scores_out, int64_t ld_scores,
    void* workspace, size_t workspace_size, void* stream) {
  return select_sharded_impl<F32>(logits, shards, rows, local_width, ld_logits, shard_stride,
                                  global_row_ks, global_row_ke, global_block_size,
                                  max_global_blocks, row_repeat, topk_blocks, out, ld_out,
                                  scores_out, ld_scores, workspace, workspace_size, stream);
}

dsa_status dsa_select_candidate_blocks_sharded_starts_bf16(
    const uint16_t* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ks, const int32_t* global_row_ke,
    int32_t global_block_size, int32_t max_global_blocks, int32_t row_repeat,
    int32_t topk_blocks, int32_t* out, int64_t ld_out, uint16_t* scores_out, int64_t ld_scores,
    void* workspace, size_t workspace_size, void* stream) {
  return select_sharded_impl<BF16>(logits, shards, rows, local_width, ld_logits, shard_stride,
                                   global_row_ks, global_row_ke, global_block_size,
                                   max_global_blocks, row_repeat, topk_blocks, out, ld_out,
                                   scores_out, ld_scores, workspace, workspace_size, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point
// ---------------------------------------------------------------------------
//
// dsa_select_candidate_blocks_sharded_static: the sharded selection with its
// workspace taken from a fixed array in device memory that this library
// declares at file scope, for callers that must not allocate device memory at
// call time. Examples: serving engines whose memory planner reserves nearly
// all of HBM (KV cache pools) at start-up, so that a cudaMalloc in the middle
// of a step can fail or block on the allocator; and plugin hosts whose
// operators may not allocate behind the host framework's back.
//
// The array (kStaticScratchBytes) is created when the library's device code
// is loaded on a GPU and stays there until the process exits; every call on
// that GPU shares it. In host code the array's name is only a host-side
// stand-in, so every call looks up its device address with
// cudaGetSymbolAddress, with the call's device current (a lookup is cheap, and
// nothing cached can go stale when a context is torn down and rebuilt).

namespace dsa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

}  // namespace
}  // namespace dsa

// Host memory that the GPU reads in place: page-locked memory is mapped into
// the device's address space (across NVLink-C2C on Grace systems), so a
// kernel can be handed its device address instead of a device copy.
extern "C" dsa_status dsa_mapped_host_pointer(const void* host, void** device) {
  if (!host || !device) return DSA_EINVAL;
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
    cudaGetLastError();  // the lookup's error is not sticky: clear it
    return DSA_EINVAL;
  }
  // The attributes must describe this very address (not only its
  // allocation), so that the device address maps the same byte.
  if (attr.type != cudaMemoryTypeHost || !attr.devicePointer || attr.hostPointer != host)
    return DSA_EINVAL;
  *device = attr.devicePointer;
  return DSA_OK;
}

extern "C" dsa_status dsa_select_candidate_blocks_sharded_static(
    const float* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ke, int32_t global_block_size,
    int32_t max_global_blocks, int32_t row_repeat, int32_t topk_blocks, int32_t* out,
    int64_t ld_out, float* scores_out, int64_t ld_scores, void* stream) {
  // Every argument error is returned before anything is enqueued.
  const int pre = dsa::sharded_precheck(logits, shards, rows, local_width, ld_logits,
                                        shard_stride, global_row_ke, global_block_size,
                                        max_global_blocks, row_repeat, topk_blocks, out, ld_out,
                                        scores_out, ld_scores);
  if (pre < 0) return static_cast<dsa_status>(pre);
  if (pre == dsa::kNoWork) return DSA_OK;
  const int64_t nbg = max_global_blocks > 1 ? max_global_blocks : 1;
  const size_t need = dsa::workspace_bytes(rows, nbg);
  void* scratch = nullptr;
  if (need <= dsa::kStaticScratchBytes) {
    if (cudaGetSymbolAddress(&scratch, dsa::g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return DSA_ECUDA;
    }
    // The array keeps whatever the previous call left: clear the part of it
    // that must start at zero (the queue header and the arrival counters).
    if (cudaMemsetAsync(scratch, 0, dsa::ws_keys_offset(rows),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return DSA_ECUDA;
  }
  // A call whose workspace does not fit in the array runs without one: rows
  // are dealt to CTAs in a fixed order and none is split, with the same
  // results.
  return dsa_select_candidate_blocks_sharded(
      logits, shards, rows, local_width, ld_logits, shard_stride, global_row_ke,
      global_block_size, max_global_blocks, row_repeat, topk_blocks, out, ld_out, scores_out,
      ld_scores, scratch, scratch ? dsa::kStaticScratchBytes : 0, stream);
}
