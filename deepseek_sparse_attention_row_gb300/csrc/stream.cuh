// stream.cuh -- the HBM pass: windowed per-block maxima of one row range.
//
// candidate_blocks.py diff, _block_scores_kernel: a row's window [s, e) is cut
// into blocks of block_size columns counted from s; each block's score is the
// NaN-propagating max of its in-window logits, -inf when it has none. In the
// DCP form a row is held as `shards` interleave-1 slices, shard d's window is
// its first len[d] local columns, local block b of every shard belongs to
// global block b, and the global score is the max over shards.
//
// Both forms are the same loop. A CTA owns block range [b0, b1) of one row
// and accumulates order keys (keys.cuh) into keys[b - kbase] in shared
// memory, initialised by the caller to key(-inf). A warp streams a slab of
// 32 x NV vectors of VEC floats per shard, lane l taking vectors l, l + 32,
// ..., so every load instruction is one contiguous, fully coalesced warp
// access; all NV x SB loads of a slab are issued before any is used, and a
// lane folds everything it loaded for one vector slot (over shards and
// vector elements) with max.NaN before anything crosses lanes. Vector v of a
// shard covers local elements [v*VEC, v*VEC + VEC) and lies in block
// v / LPB, LPB = block_size / VEC.
//
// Fast path (stream_pow2): VEC divides block_size, LPB is a power of two and
// every shard origin is VEC*4-byte aligned. With LPB <= 32 a load
// instruction covers 32 / LPB whole blocks: log2(LPB) xor-shuffles reduce a
// block and its first lane stores the key. With LPB > 32 the instructions of
// one block are folded in registers first, then one redux.sync and one
// shared atomicMax per block and slab. Generic path (stream_generic): scalar
// loads, a block id per lane, a segmented shuffle reduction and an atomicMax
// per block segment.
//
// No element outside a window is read. The hot loop loads only whole vectors
// inside the window; the one vector per shard that straddles the window end
// is read element by element by load_partial().
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

template <typename E>
struct Window {
  const typename E::T* origin;  // element 0 of shard 0's window
  int64_t shard_stride;  // elements between shards
  int32_t shards;
  const int32_t* len;    // shared memory: in-window length of each shard
  int32_t len_max;       // max over shards of len[d]
  bool merge = false;    // keys may already hold other data: merge with atomicMax
};

// Fast path. lpb_log2 = log2(block_size / VEC).
// Warp `warp` of `nwarps` warps working on the range (a whole CTA: the CTA's
// warp index and count; one warp alone: 0 and 1).
template <typename E, int VEC, int NV, int SB>
__device__ __forceinline__ void stream_pow2(const Window<E>& w, int lpb_log2, int32_t b0, int32_t b1,
                                            uint32_t* __restrict__ keys, int32_t kbase, int warp,
                                            int nwarps) {
  const int lane = threadIdx.x & 31;
  const int lpb = 1 << lpb_log2;
  const int32_t nvec = w.len_max / VEC;  // whole vectors of the longest shard
  const int32_t v_begin = static_cast<int32_t>(static_cast<int64_t>(b0) << lpb_log2);
  const int32_t v_end = static_cast<int32_t>(min(static_cast<int64_t>(b1) << lpb_log2,
                                                 static_cast<int64_t>(nvec)));
  // Several shard batches commit to the same blocks: merge with atomics.
  const bool merge = w.shards > SB || w.merge;
  constexpr int32_t kSlab = 32 * NV;

  for (int d0 = 0; d0 < w.shards; d0 += SB) {
    int32_t lim[SB];
    int32_t lim_min = v_end;  // slabs below it lie inside every shard's window
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      lim[j] = (d0 + j < w.shards) ? min(w.len[d0 + j] / VEC, v_end) : 0;
      lim_min = min(lim_min, lim[j]);
    }
    const typename E::T* base = w.origin + static_cast<int64_t>(d0) * w.shard_stride;

    const int32_t step = nwarps * kSlab;
    for (int32_t slab = v_begin + warp * kSlab; slab < v_end; slab += step) {
      float acc[NV];
#pragma unroll
      for (int m = 0; m < NV; ++m) acc[m] = neg_inf();
      Raw<E, VEC> x[SB][NV];
      if (slab + kSlab <= lim_min) {
        // A full slab: every load is inside its shard's window.
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          const typename E::T* src = base + static_cast<int64_t>(j) * w.shard_stride;
#pragma unroll
          for (int m = 0; m < NV; ++m)
            ld_raw<E, VEC>(src + static_cast<int64_t>(slab + m * 32 + lane) * VEC, x[j][m]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          const typename E::T* src = base + static_cast<int64_t>(j) * w.shard_stride;
#pragma unroll
          for (int m = 0; m < NV; ++m) {
            const int32_t v = slab + m * 32 + lane;
            if (v < lim[j])
              ld_raw<E, VEC>(src + static_cast<int64_t>(v) * VEC, x[j][m]);
            else
              raw_neg_inf(x[j][m]);
          }
        }
      }
      if constexpr (E::kBytes == 2 && VEC >= 2) {
        // bf16 pairs: fold every word of the slot with the packed
        // max.NaN.bf16x2 (the same total order in each half), then widen the
        // two halves once.
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          uint32_t a2 = x[0][m].w[0];
#pragma unroll
          for (int j = 0; j < SB; ++j)
#pragma unroll
            for (int i = (j == 0 ? 1 : 0); i < Raw<E, VEC>::kWords; ++i)
              a2 = max_nan_bf16x2(a2, x[j][m].w[i]);
          acc[m] = max_nan(__uint_as_float(a2 << 16), __uint_as_float(a2 & 0xFFFF0000u));
        }
      } else {
#pragma unroll
        for (int j = 0; j < SB; ++j)
#pragma unroll
          for (int m = 0; m < NV; ++m) acc[m] = fold(acc[m], x[j][m]);
      }

      if (lpb_log2 >= 5) {
        // Instructions m of one block are consecutive; fold them, then one
        // warp reduction per block.
        float carry = neg_inf();
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          carry = max_nan(carry, acc[m]);
          const int32_t blk = (slab + m * 32) >> lpb_log2;
          const bool last = (m == NV - 1) || (((slab + (m + 1) * 32) >> lpb_log2) != blk);
          if (last) {
            if (blk < b1) {
              const uint32_t k = __reduce_max_sync(0xffffffffu, order_key(carry));
              if (lane == 0) atomicMax(&keys[blk - kbase], k);
            }
            carry = neg_inf();
          }
        }
      } else {
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int32_t vfirst = slab + m * 32;
          if (vfirst >= v_end) break;
          uint32_t k = order_key(acc[m]);
          for (int o = 1; o < lpb; o <<= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
          const int32_t v = vfirst + lane;
          if ((lane & (lpb - 1)) == 0 && v < v_end) {
            if (merge)
              atomicMax(&keys[(v >> lpb_log2) - kbase], k);
            else
              keys[(v >> lpb_log2) - kbase] = k;
          }
        }
      }
    }
  }
}

// One unsharded window whose start lies r = 1..VEC-1 elements past a 16-byte
// boundary (the same layout as stream_shift below, one row): each lane folds
// a hi and a lo part per vector, and a lead vector's lo part is merged into
// the block before with atomicMax; the hi parts reduce per block and merge
// with atomicMax. Measured on GB300 against the shuffle merge of
// stream_shift with one shard: equal on prefill-like rows, and faster on
// long rows and for the rest of the kernel (decode rows do not use it but
// share the kernel's registers).
template <typename E, int NV>
__device__ __forceinline__ void stream_shift_row(const typename E::T* origin, int32_t r,
                                                 int32_t len, int lpb_log2, int32_t b0, int32_t b1,
                                                 uint32_t* __restrict__ keys, int32_t kbase,
                                                 int warp, int nwarps) {
  constexpr int VEC = 16 / E::kBytes;
  const int lane = threadIdx.x & 31;
  const int lpb = 1 << lpb_log2;
  const typename E::T* base = origin - r;
  const int32_t nvec = (len + r) / VEC;  // whole vectors of base inside [base, origin + len)
  const int32_t v_begin = static_cast<int32_t>(static_cast<int64_t>(b0) << lpb_log2);
  const int32_t v_end = static_cast<int32_t>(min((static_cast<int64_t>(b1) << lpb_log2) + 1,
                                                 static_cast<int64_t>(nvec)));
  constexpr int32_t kSlab = 32 * NV;
  const int32_t step = nwarps * kSlab;
  for (int32_t slab = v_begin + warp * kSlab; slab < v_end; slab += step) {
    Raw<E, VEC> x[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int32_t v = slab + m * 32 + lane;
      if (v < v_end)
        ld_raw<E, VEC>(base + static_cast<int64_t>(v) * VEC, x[m]);
      else
        raw_neg_inf(x[m]);
    }
    float hi[NV], lo[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int32_t v = slab + m * 32 + lane;
      const bool lead = (v & (lpb - 1)) == 0;
      hi[m] = neg_inf();
      lo[m] = neg_inf();
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const bool below = lead && i < r;
        const float xi = raw_elem(x[m], i);
        hi[m] = max_nan(hi[m], below ? neg_inf() : xi);
        lo[m] = max_nan(lo[m], below ? xi : neg_inf());
      }
    }
    // lo parts: the lead lane of each block sends them to the block before.
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int32_t v = slab + m * 32 + lane;
      const int32_t blk = (v >> lpb_log2) - 1;
      if ((v & (lpb - 1)) == 0 && v < v_end && blk >= b0 && blk < b1)
        atomicMax(&keys[blk - kbase], order_key(lo[m]));
    }
    // hi parts, reduced per block as in the aligned path.
    if (lpb_log2 >= 5) {
      float carry = neg_inf();
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        carry = max_nan(carry, hi[m]);
        const int32_t blk = (slab + m * 32) >> lpb_log2;
        const bool last = (m == NV - 1) || (((slab + (m + 1) * 32) >> lpb_log2) != blk);
        if (last) {
          if (blk < b1) {
            const uint32_t k = __reduce_max_sync(0xffffffffu, order_key(carry));
            if (lane == 0) atomicMax(&keys[blk - kbase], k);
          }
          carry = neg_inf();
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        const int32_t vfirst = slab + m * 32;
        if (vfirst >= v_end) break;
        uint32_t k = order_key(hi[m]);
        for (int o = 1; o < lpb; o <<= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
        const int32_t v = vfirst + lane;
        const int32_t blk = v >> lpb_log2;
        if ((lane & (lpb - 1)) == 0 && v < v_end && blk < b1) atomicMax(&keys[blk - kbase], k);
      }
    }
  }
}


// Shard rows of the DCP form with starts (up to two groups of shards, each
// group sharing its window start and so its offset r = 0..VEC-1 past a
// 16-byte boundary; VEC = 16-byte vector in elements, 4 fp32 or 8 bf16),
// block size a power-of-two multiple of VEC (LPB = block_size / VEC a power
// of two). Each shard loads aligned 16-byte vectors from its base
// origin - r. Vector v of a shard covers its window elements
// [VEC*v - r, VEC*v - r + VEC); all of them belong to block v / LPB except,
// in the block's first vector (v % LPB == 0), the r elements below the block
// boundary, which belong to block v / LPB - 1 (and, for v = 0, precede the
// window and are dropped). Because blocks count from each shard's own
// start, vector v maps to the same blocks in both groups: the shards of a
// group are folded element-wise, each group's vector is split at its own r
// into a "hi" value for block v / LPB and, in a block's first vector, a "lo"
// value for the block before, and the two groups' parts are combined.
// A lo value joins the hi value of vector v - 1, which the next lane down
// (or lane 31 of the previous instruction) holds, through one shuffle; only
// the lo value of a slab's first vector crosses to another warp's slab and
// is merged with atomicMax. With several blocks per instruction (LPB < 32) a
// slab's last block is therefore the one block written with atomicMax (every
// block when `merge`); larger blocks span slabs and are always merged with
// atomicMax. Vector b1 * LPB is read only for its lo part (it completes
// block b1 - 1). Elements past each shard's last whole vector are left to
// commit_partial_shifted.
template <typename E>
struct ShiftGroups {
  const typename E::T* base[2];  // aligned base of shard 0's row for each group
  int32_t r[2];                  // the groups' offsets
  int32_t split;                 // shards [0, split) belong to group 1, the rest to group 0
  int64_t shard_stride;
  int32_t shards;
  const int32_t* len;            // shared memory: in-window length of each shard
  int32_t v_cap;                 // max over shards of (len + r) / VEC
  bool merge;
};

template <typename E, int NV, int SB>
__device__ __forceinline__ void stream_shift(const ShiftGroups<E>& w, int lpb_log2, int32_t b0,
                                             int32_t b1, uint32_t* __restrict__ keys,
                                             int32_t kbase, int warp, int nwarps) {
  constexpr int VEC = 16 / E::kBytes;
  const int lane = threadIdx.x & 31;
  const int lpb = 1 << lpb_log2;
  const int32_t v_begin = static_cast<int32_t>(static_cast<int64_t>(b0) << lpb_log2);
  const int32_t v_end = static_cast<int32_t>(min((static_cast<int64_t>(b1) << lpb_log2) + 1,
                                                 static_cast<int64_t>(w.v_cap)));
  const bool merge = w.shards > SB || w.merge;
  constexpr int32_t kSlab = 32 * NV;
  const int32_t step = nwarps * kSlab;

  for (int d0 = 0; d0 < w.shards; d0 += SB) {
    int32_t lim[SB];
    const typename E::T* src[SB];
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int d = d0 + j;
      const bool g1 = d < w.split;  // constant indices keep w in registers
      lim[j] = d < w.shards ? min((w.len[d] + (g1 ? w.r[1] : w.r[0])) / VEC, v_end) : 0;
      src[j] = (g1 ? w.base[1] : w.base[0]) + static_cast<int64_t>(d) * w.shard_stride;
    }

    for (int32_t slab = v_begin + warp * kSlab; slab < v_end; slab += step) {
      Raw<E, VEC> x[SB][NV];
#pragma unroll
      for (int j = 0; j < SB; ++j) {
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int32_t v = slab + m * 32 + lane;
          if (v < lim[j])
            ld_raw<E, VEC>(src[j] + static_cast<int64_t>(v) * VEC, x[j][m]);
          else
            raw_neg_inf(x[j][m]);
        }
      }
      float hi[NV], lo[NV];
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        // Element-wise max over each group's shards, then one split per group.
        Raw<E, VEC> e[2];
        raw_neg_inf(e[0]);
        raw_neg_inf(e[1]);
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          if (d0 + j < w.split)
            raw_max(e[1], x[j][m]);
          else
            raw_max(e[0], x[j][m]);
        }
        const int32_t v = slab + m * 32 + lane;
        const bool lead = (v & (lpb - 1)) == 0;
        hi[m] = neg_inf();
        lo[m] = neg_inf();
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const float x0 = raw_elem(e[0], i), x1 = raw_elem(e[1], i);
          const bool below0 = lead && i < w.r[0], below1 = lead && i < w.r[1];
          hi[m] = max_nan(hi[m], below0 ? neg_inf() : x0, below1 ? neg_inf() : x1);
          lo[m] = max_nan(lo[m], below0 ? x0 : neg_inf(), below1 ? x1 : neg_inf());
        }
      }
      // The slab's first vector sends its lo part to the block before
      // (another slab's) with an atomic; every other lo part joins the hi
      // part one vector down.
      if (lane == 0) {
        const int32_t blk = (slab >> lpb_log2) - 1;
        if ((slab & (lpb - 1)) == 0 && blk >= b0 && blk < b1)
          atomicMax(&keys[blk - kbase], order_key(lo[0]));
      }
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        float nxt = __shfl_down_sync(0xffffffffu, lo[m], 1);
        const float first_of_next =
            __shfl_sync(0xffffffffu, m + 1 < NV ? lo[m + 1 < NV ? m + 1 : m] : neg_inf(), 0);
        if (lane == 31) nxt = first_of_next;
        hi[m] = max_nan(hi[m], nxt);
      }
      if (lpb_log2 >= 5) {
        // A block spans whole instructions (and maybe slabs): fold, then one
        // warp reduction and one atomicMax per block and slab.
        float carry = neg_inf();
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          carry = max_nan(carry, hi[m]);
          const int32_t blk = (slab + m * 32) >> lpb_log2;
          const bool last = (m == NV - 1) || (((slab + (m + 1) * 32) >> lpb_log2) != blk);
          if (last) {
            if (blk < b1) {
              const uint32_t k = __reduce_max_sync(0xffffffffu, order_key(carry));
              if (lane == 0) atomicMax(&keys[blk - kbase], k);
            }
            carry = neg_inf();
          }
        }
      } else {
        // Several blocks per instruction: one reduction per block; only a
        // slab's last block can also receive a lo part from another slab.
        const int32_t last_blk = (slab + kSlab - 1) >> lpb_log2;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int32_t vfirst = slab + m * 32;
          if (vfirst >= v_end) break;
          uint32_t k = order_key(hi[m]);
          for (int o = 1; o < lpb; o <<= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
          const int32_t v = vfirst + lane;
          const int32_t blk = v >> lpb_log2;
          if ((lane & (lpb - 1)) == 0 && v < v_end && blk < b1) {
            if (merge || blk == last_blk)
              atomicMax(&keys[blk - kbase], k);
            else
              keys[blk - kbase] = k;
          }
        }
      }
    }
  }
}

// The DCP form with starts, both shard groups read from ONE aligned base.
// With gs = q * shards + rg, shards d < rg (group 1) start at local column
// q + 1 and the others (group 0) at q; every shard row is read from column
// q - r0, r0 = q's offset past a 16-byte boundary (0 <= r0 < VEC). Window
// element t of a group-g shard then sits at stream position t + r0 + g, in
// block (t) / block_size. For stream position p = VEC*v + i the two groups
// put element i in the same block unless p - r0 is a multiple of the block
// size, i.e. unless v is a block's first vector (v % LPB == 0) and i = r0:
// there group 0 starts block v / LPB while group 1 ends block v / LPB - 1.
// So a lane folds its 16-byte vectors of all shards element-wise (no group
// routing), splits the result at r0 into a "lo" part (the block before) and
// a "hi" part, and routes only element r0 by group: the group-0 maximum of
// that element joins hi, the group-1 maximum joins lo. Vectors past a
// shard's window load as -inf (only in the slab that crosses the shortest
// shard's end; full slabs load unconditionally). lo and hi then meet as in
// stream_shift: lo joins the hi of the vector below (one shuffle), a slab's
// first lo goes to the previous slab's block with atomicMax, and a slab's
// last block is written with atomicMax. Elements past each shard's last
// whole vector are left to commit_partial_shifted.
template <typename E>
struct PairedShift {
  const typename E::T* base;  // shard 0's row at column q - r0 (16-byte aligned)
  int32_t r0;                 // 0 .. VEC-1
  int32_t split;              // shards [0, split) belong to group 1
  int64_t shard_stride;
  int32_t shards;
  const int32_t* len;         // shared memory: in-window length of each shard
  int32_t v_cap;              // max over shards of (len + r0 + group) / VEC
  bool merge;
};

template <typename E, int SB>
__device__ __forceinline__ void stream_shift_paired(const PairedShift<E>& w, int lpb_log2,
                                                    int32_t b0, int32_t b1,
                                                    uint32_t* __restrict__ keys, int32_t kbase,
                                                    int warp, int nwarps) {
  constexpr int VEC = 16 / E::kBytes;
  const int lane = threadIdx.x & 31;
  const int lpb = 1 << lpb_log2;
  const int32_t v_begin = static_cast<int32_t>(static_cast<int64_t>(b0) << lpb_log2);
  const int32_t v_end = static_cast<int32_t>(min((static_cast<int64_t>(b1) << lpb_log2) + 1,
                                                 static_cast<int64_t>(w.v_cap)));
  const bool merge = w.shards > SB || w.merge;
  const int r0 = w.r0;
  constexpr int32_t kSlab = 32;
  const int32_t step = nwarps * kSlab;

  for (int d0 = 0; d0 < w.shards; d0 += SB) {
    int32_t lim[SB];
    bool g1[SB];
    // Shard j of the batch is read at row0 + j * shard_stride (no pointer per
    // shard held across the loop).
    const typename E::T* row0 = w.base + static_cast<int64_t>(d0) * w.shard_stride;
    int32_t lim_min = v_end;
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int d = d0 + j;
      g1[j] = d < w.split;
      const int32_t n = d < w.shards ? w.len[d] : 0;
      lim[j] = n > 0 ? min((n + r0 + (g1[j] ? 1 : 0)) / VEC, v_end) : 0;
      if (d < w.shards) lim_min = min(lim_min, lim[j]);
    }
    // In the last batch, shards past the end load nothing.
    if (d0 + SB > w.shards) lim_min = 0;

    for (int32_t slab = v_begin + warp * kSlab; slab < v_end; slab += step) {
      const int32_t v = slab + lane;
      const typename E::T* at = row0 + static_cast<int64_t>(v) * VEC;
      Raw<E, VEC> x[SB];
      if (slab + kSlab <= lim_min) {
#pragma unroll
        for (int j = 0; j < SB; ++j) ld_raw<E, VEC>(at + j * w.shard_stride, x[j]);
      } else {
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          if (v < lim[j])
            ld_raw<E, VEC>(at + j * w.shard_stride, x[j]);
          else
            raw_neg_inf(x[j]);
        }
      }
      // Element-wise max over every shard (three-operand max for fp32, the
      // packed bf16 pair max for bf16), and element r0 by group.
      float ae[VEC];
      if constexpr (E::kBytes == 4) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          float m = __uint_as_float(x[0].w[i]);
#pragma unroll
          for (int j = 1; j < SB; j += 2)
            m = j + 1 < SB ? max_nan(m, __uint_as_float(x[j].w[i]), __uint_as_float(x[j + 1].w[i]))
                           : max_nan(m, __uint_as_float(x[j].w[i]));
          ae[i] = m;
        }
      } else {
        Raw<E, VEC> a = x[0];
#pragma unroll
        for (int j = 1; j < SB; ++j) raw_max(a, x[j]);
#pragma unroll
        for (int i = 0; i < VEC; ++i) ae[i] = raw_elem(a, i);
      }
      float xr[SB];
#pragma unroll
      for (int j = 0; j < SB; ++j) xr[j] = raw_elem_at(x[j], r0);
      float gr0 = neg_inf(), gr1 = neg_inf();
#pragma unroll
      for (int j = 0; j < SB; j += 2) {
        if (j + 1 < SB) {
          gr1 = max_nan(gr1, g1[j] ? xr[j] : neg_inf(), g1[j + 1] ? xr[j + 1] : neg_inf());
          gr0 = max_nan(gr0, g1[j] ? neg_inf() : xr[j], g1[j + 1] ? neg_inf() : xr[j + 1]);
        } else {
          gr1 = max_nan(gr1, g1[j] ? xr[j] : neg_inf());
          gr0 = max_nan(gr0, g1[j] ? neg_inf() : xr[j]);
        }
      }
      float lo = neg_inf(), hi = neg_inf(), all = neg_inf();
#pragma unroll
      for (int i = 0; i < VEC; i += 2) {
        all = max_nan(all, ae[i], ae[i + 1]);
        lo = max_nan(lo, i < r0 ? ae[i] : neg_inf(), i + 1 < r0 ? ae[i + 1] : neg_inf());
        hi = max_nan(hi, i > r0 ? ae[i] : neg_inf(), i + 1 > r0 ? ae[i + 1] : neg_inf());
      }
      const bool lead = (v & (lpb - 1)) == 0;
      hi = lead ? max_nan(hi, gr0) : all;
      lo = lead ? max_nan(lo, gr1) : neg_inf();
      // The slab's first vector sends its lo part to the block before (in
      // another warp's slab) with an atomic; every other lo part joins the
      // hi part of the vector below it.
      if (lane == 0) {
        const int32_t blk = (slab >> lpb_log2) - 1;
        if ((slab & (lpb - 1)) == 0 && blk >= b0 && blk < b1)
          atomicMax(&keys[blk - kbase], order_key(lo));
      }
      float nxt = __shfl_down_sync(0xffffffffu, lo, 1);
      if (lane == 31) nxt = neg_inf();
      hi = max_nan(hi, nxt);
      if (lpb_log2 >= 5) {
        // A block spans whole slabs: one warp reduction and one atomicMax per
        // block and slab.
        const int32_t blk = slab >> lpb_log2;
        if (blk < b1) {
          const uint32_t k = __reduce_max_sync(0xffffffffu, order_key(hi));
          if (lane == 0) atomicMax(&keys[blk - kbase], k);
        }
      } else {
        // Several blocks per slab: one reduction per block; only the slab's
        // last block can also receive a lo part from another slab.
        const int32_t last_blk = (slab + kSlab - 1) >> lpb_log2;
        uint32_t k = order_key(hi);
        for (int o = 1; o < lpb; o <<= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
        const int32_t blk = v >> lpb_log2;
        if ((lane & (lpb - 1)) == 0 && v < v_end && blk < b1) {
          if (merge || blk == last_blk)
            atomicMax(&keys[blk - kbase], k);
          else
            keys[blk - kbase] = k;
        }
      }
    }
  }
}

// Elements of a shifted window (stream_shift) past its last whole vector:
// window elements [VEC * nvec - r, len), each to its own block (the run can
// cross one block boundary). One thread; call after the loop and a barrier.
template <typename E>
__device__ __forceinline__ void commit_partial_shifted(const typename E::T* origin, int32_t r,
                                                       int32_t len, int32_t block_size,
                                                       int32_t b0, int32_t b1, uint32_t* keys,
                                                       int32_t kbase) {
  constexpr int VEC = 16 / E::kBytes;
  const int32_t first = max(((len + r) / VEC) * VEC - r, 0);
  const bool pow2 = (block_size & (block_size - 1)) == 0;
  const int sh = __ffs(block_size) - 1;
  for (int32_t i = first; i < len; ++i) {
    const int32_t blk = pow2 ? (i >> sh) : i / block_size;
    if (blk >= b0 && blk < b1) atomicMax(&keys[blk - kbase], order_key(ld_elem(origin + i)));
  }
}

// The elements past the last whole vector of a shard's window (at most
// VEC - 1) are read after the streaming loop: load_partial() folds them into
// a register and commit_partial() merges that into their block, after a
// __syncthreads() (the loop stores keys without atomics). Loading them before
// the loop instead measured slower (the live registers cost the loop).
struct Partial {
  float v;
  int32_t blk;  // -1: nothing to merge
};

template <typename E, int VEC>
__device__ __forceinline__ Partial load_partial(const typename E::T* shard_origin, int32_t len,
                                                int32_t block_size, int32_t b0, int32_t b1) {
  Partial p{neg_inf(), -1};
  if (VEC == 1) return p;
  const int32_t first = (len / VEC) * VEC;
  if (first == len) return p;
  const int32_t blk = (block_size & (block_size - 1)) == 0 ? first >> (__ffs(block_size) - 1)
                                                           : first / block_size;
  if (blk < b0 || blk >= b1) return p;
  for (int32_t i = first; i < len; ++i) p.v = max_nan(p.v, ld_elem(shard_origin + i));
  p.blk = blk;
  return p;
}

__device__ __forceinline__ void commit_partial(const Partial& p, uint32_t* keys, int32_t kbase) {
  if (p.blk >= 0) atomicMax(&keys[p.blk - kbase], order_key(p.v));
}

// Generic path: any block size, any alignment. Elements, not vectors.
template <typename E, int NV, int SB>
__device__ __forceinline__ void stream_generic(const Window<E>& w, int32_t block_size, int32_t b0,
                                               int32_t b1, uint32_t* __restrict__ keys,
                                               int32_t kbase, int warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  const int64_t e_begin = static_cast<int64_t>(b0) * block_size;
  const int64_t e_end = min(static_cast<int64_t>(b1) * block_size, static_cast<int64_t>(w.len_max));
  constexpr int64_t kSlab = 32 * NV;

  const int64_t step = static_cast<int64_t>(nwarps) * kSlab;
  for (int64_t slab = e_begin + warp * kSlab; slab < e_end; slab += step) {
    float acc[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) acc[m] = neg_inf();
    for (int d0 = 0; d0 < w.shards; d0 += SB) {
      float x[SB][NV];
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        const int32_t len = (d0 + j < w.shards) ? w.len[d0 + j] : 0;
        const typename E::T* src = w.origin + static_cast<int64_t>(d0 + j) * w.shard_stride;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int64_t i = slab + m * 32 + lane;
          x[j][m] = (i < e_end && i < len) ? ld_elem(src + i) : neg_inf();
        }
      }
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int m = 0; m < NV; ++m) acc[m] = max_nan(acc[m], x[j][m]);
    }
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int64_t first = slab + m * 32;
      if (first >= e_end) break;
      const int64_t i = first + lane;
      const int32_t blk = (i < e_end) ? static_cast<int32_t>(i / block_size) : -1;
      uint32_t k = order_key(acc[m]);
      // Segmented max over runs of equal blk (runs are contiguous in lanes):
      // afterwards the first lane of each run holds the run's max.
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t ok = __shfl_down_sync(0xffffffffu, k, o);
        const int32_t ob = __shfl_down_sync(0xffffffffu, blk, o);
        if (lane + o < 32 && ob == blk) k = max(k, ok);
      }
      const int32_t prev = __shfl_up_sync(0xffffffffu, blk, 1);
      if (blk >= 0 && (lane == 0 || prev != blk)) atomicMax(&keys[blk - kbase], k);
    }
  }
}

// Per-row choice of the vector width (elements) for a window origin
// (unsharded rows start at arbitrary columns): the widest of 16, 8, 4 (and,
// for bf16, 2) bytes that the origin's alignment allows and that splits the
// block into a power of two of vectors. Returns 0 for the generic path.
template <typename E>
__device__ __forceinline__ int choose_vec(const typename E::T* origin, int32_t block_size,
                                          int* lpb_log2) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(origin);
  auto pow2 = [](int32_t x) { return x > 0 && (x & (x - 1)) == 0; };
  int vec = 0;
  for (int bytes = 16; bytes >= 2 * E::kBytes; bytes >>= 1) {
    const int v = bytes / E::kBytes;
    if (block_size % v == 0 && (a & (bytes - 1)) == 0 && pow2(block_size / v)) {
      vec = v;
      break;
    }
  }
  if (!vec && pow2(block_size)) vec = 1;
  *lpb_log2 = vec ? __ffs(block_size / vec) - 1 : 0;
  return vec;
}

// Unsharded dispatch: vector width chosen per row at run time. Every path
// keeps 32 words per lane in flight per slab.
// kVecShift: shifted 16-byte loads (stream_shift) for a window starting
// `shift` elements past a 16-byte boundary (no element count is this large).
constexpr int kVecShift = 64;

template <typename E>
__device__ __forceinline__ void stream_row(const Window<E>& w, int vec, int shift, int lpb_log2,
                                           int32_t block_size, int32_t b0, int32_t b1,
                                           uint32_t* keys, int32_t kbase, int warp, int nwarps) {
  constexpr int V16 = 16 / E::kBytes;  // elements per 16 / 8 / 4-byte vector
  constexpr int V8 = 8 / E::kBytes;
  constexpr int V4 = 4 / E::kBytes;
  if (vec == kVecShift)
    stream_shift_row<E, 8>(w.origin, shift, w.len_max, lpb_log2, b0, b1, keys, kbase, warp,
                           nwarps);
  else if (vec == V16)
    stream_pow2<E, V16, 8, 1>(w, lpb_log2, b0, b1, keys, kbase, warp, nwarps);
  else if (vec == V8)
    stream_pow2<E, V8, 16, 1>(w, lpb_log2, b0, b1, keys, kbase, warp, nwarps);
  else if (vec == V4 && V4 > 1)
    stream_pow2<E, (V4 > 1 ? V4 : 2), 32, 1>(w, lpb_log2, b0, b1, keys, kbase, warp, nwarps);
  else if (vec == 1)
    stream_pow2<E, 1, 32, 1>(w, lpb_log2, b0, b1, keys, kbase, warp, nwarps);
  else
    stream_generic<E, 16, 1>(w, block_size, b0, b1, keys, kbase, warp, nwarps);
}

// Tail of an unsharded row past its last whole vector; one thread, after the
// loop and a barrier.
template <typename E>
__device__ __forceinline__ void finish_row(const Window<E>& w, int vec, int shift,
                                           int32_t block_size, int32_t b0, int32_t b1,
                                           uint32_t* keys, int32_t kbase) {
  constexpr int V16 = 16 / E::kBytes;
  constexpr int V8 = 8 / E::kBytes;
  constexpr int V4 = 4 / E::kBytes;
  if (vec == V16)
    commit_partial(load_partial<E, V16>(w.origin, w.len_max, block_size, b0, b1), keys, kbase);
  else if (vec == V8)
    commit_partial(load_partial<E, V8>(w.origin, w.len_max, block_size, b0, b1), keys, kbase);
  else if (vec == V4 && V4 > 1)
    commit_partial(load_partial<E, (V4 > 1 ? V4 : 2)>(w.origin, w.len_max, block_size, b0, b1),
                   keys, kbase);
  else if (vec == kVecShift)
    commit_partial_shifted<E>(w.origin, shift, w.len_max, block_size, b0, b1, keys, kbase);
}

}  // namespace dsa
