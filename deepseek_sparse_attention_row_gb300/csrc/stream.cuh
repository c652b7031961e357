// stream.cuh -- the HBM pass: windowed per-block maxima of one row range.
//
// candidate_blocks.py diff, _block_scores_kernel: a row's window [s, e) is cut
// into blocks of block_size columns counted from s; each block's score is the
// NaN-propagating max of its in-window logits, -inf when it has none. In the
// DCP form a row is held as `shards` interleave-1 slices, shard d's window is
// its first len[d] local columns, local block b of every shard belongs to
// global block b, and the global score is the max over shards.
//
// Both forms are the same loop here. Each CTA owns block range [b0, b1) of
// one row and accumulates order keys (keys.cuh) into keys[b - kbase] in shared
// memory, which the caller initialised to key(-inf). A warp streams a slab of
// 32 x NV vectors of VEC floats per shard, lane l taking vectors l, l + 32, ...
// so every load instruction is a contiguous, fully coalesced warp access; all
// NV x SB loads of a slab are issued before any is used. Vector v of a shard
// covers local elements [v*VEC, v*VEC + VEC) and lies in block
// v / (block_size / VEC).
//
// Fast path (stream_pow2): VEC divides block_size, LPB = block_size / VEC is
// a power of two, and every shard's origin is VEC*4-byte aligned. With
// LPB <= 32 a load instruction covers 32 / LPB whole blocks, reduced by
// log2(LPB) xor-shuffles and stored by the group's first lane; with LPB > 32
// it covers part of one block, reduced with redux.sync and merged by a shared
// atomicMax. Generic path (stream_generic): scalar loads, block id per lane,
// a segmented shuffle reduction and an atomicMax per block segment.
//
// No element outside a window is read: full vectors are loaded only when
// they lie inside the window, and the one partial vector per shard at the
// window end is read element by element.
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct Window {
  const float* origin;   // element 0 of shard 0's window
  int64_t shard_stride;  // elements between shards (0 when shards == 1)
  int32_t shards;
  const int32_t* len;    // shared memory: in-window length of each shard
  int32_t len_max;       // max over shards of len[d]
};

template <int VEC>
__device__ __forceinline__ void fill_neg(float (&x)[VEC]) {
#pragma unroll
  for (int i = 0; i < VEC; ++i) x[i] = __uint_as_float(0xFF800000u);  // -inf
}

template <int VEC>
__device__ __forceinline__ uint32_t vec_key(const float (&x)[VEC]) {
  uint32_t k = order_key(x[0]);
#pragma unroll
  for (int i = 1; i < VEC; ++i) k = max(k, order_key(x[i]));
  return k;
}

// Fast path. lpb_log2 = log2(block_size / VEC).
template <int VEC, int NV, int SB>
__device__ __forceinline__ void stream_pow2(const Window& w, int lpb_log2, int32_t b0, int32_t b1,
                                            uint32_t* __restrict__ keys, int32_t kbase) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int lpb = 1 << lpb_log2;
  const int64_t nvec = (static_cast<int64_t>(w.len_max) + VEC - 1) / VEC;
  const int64_t v_begin = static_cast<int64_t>(b0) << lpb_log2;
  const int64_t v_end = min(static_cast<int64_t>(b1) << lpb_log2, nvec);
  constexpr int64_t kSlab = 32 * NV;

  for (int64_t slab = v_begin + warp * kSlab; slab < v_end; slab += kWarps * kSlab) {
    uint32_t key[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) key[m] = kKeyNegInf;

    for (int d0 = 0; d0 < w.shards; d0 += SB) {
      float x[SB][NV][VEC];
      int32_t len[SB];
#pragma unroll
      for (int j = 0; j < SB; ++j) len[j] = (d0 + j < w.shards) ? w.len[d0 + j] : 0;
      // Issue every full-vector load of the slab first.
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        const float* src = w.origin + static_cast<int64_t>(d0 + j) * w.shard_stride;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int64_t v = slab + m * 32 + lane;
          if (v < v_end && (v + 1) * VEC <= len[j])
            ld_stream(src + v * VEC, x[j][m]);
          else
            fill_neg<VEC>(x[j][m]);
        }
      }
      // The vector that straddles a shard's window end (at most one per
      // shard) is read element by element.
      if (VEC > 1) {
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          const float* src = w.origin + static_cast<int64_t>(d0 + j) * w.shard_stride;
#pragma unroll
          for (int m = 0; m < NV; ++m) {
            const int64_t v = slab + m * 32 + lane;
            if (v < v_end && v * VEC < len[j] && (v + 1) * VEC > len[j]) {
#pragma unroll
              for (int i = 0; i < VEC; ++i)
                if (v * VEC + i < len[j]) x[j][m][i] = ld_stream1(src + v * VEC + i);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int m = 0; m < NV; ++m) key[m] = max(key[m], vec_key<VEC>(x[j][m]));
    }

    // Reduce each load instruction's 32 vectors to block keys and commit.
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int64_t vfirst = slab + m * 32;
      if (vfirst >= v_end) break;
      uint32_t k = key[m];
      if (lpb_log2 >= 5) {
        k = __reduce_max_sync(0xffffffffu, k);
        if (lane == 0) atomicMax(&keys[static_cast<int32_t>(vfirst >> lpb_log2) - kbase], k);
      } else {
        for (int o = 1; o < lpb; o <<= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
        const int64_t v = vfirst + lane;
        if ((lane & (lpb - 1)) == 0 && v < v_end)
          keys[static_cast<int32_t>(v >> lpb_log2) - kbase] = k;
      }
    }
  }
}

// Generic path: any block size, any alignment. Elements, not vectors.
template <int NV, int SB>
__device__ __forceinline__ void stream_generic(const Window& w, int32_t block_size, int32_t b0,
                                               int32_t b1, uint32_t* __restrict__ keys,
                                               int32_t kbase) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t e_begin = static_cast<int64_t>(b0) * block_size;
  const int64_t e_end = min(static_cast<int64_t>(b1) * block_size, static_cast<int64_t>(w.len_max));
  constexpr int64_t kSlab = 32 * NV;

  for (int64_t slab = e_begin + warp * kSlab; slab < e_end; slab += kWarps * kSlab) {
    uint32_t key[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) key[m] = kKeyNegInf;
    for (int d0 = 0; d0 < w.shards; d0 += SB) {
      float x[SB][NV];
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        const int32_t len = (d0 + j < w.shards) ? w.len[d0 + j] : 0;
        const float* src = w.origin + static_cast<int64_t>(d0 + j) * w.shard_stride;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const int64_t i = slab + m * 32 + lane;
          x[j][m] = (i < e_end && i < len) ? ld_stream1(src + i) : __uint_as_float(0xFF800000u);
        }
      }
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int m = 0; m < NV; ++m) key[m] = max(key[m], order_key(x[j][m]));
    }
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int64_t first = slab + m * 32;
      if (first >= e_end) break;
      const int64_t i = first + lane;
      const int32_t blk = (i < e_end) ? static_cast<int32_t>(i / block_size) : -1;
      uint32_t k = key[m];
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

// Per-row choice of the vector width for a window origin (unsharded rows
// start at arbitrary columns). Returns 0 for the generic path.
__device__ __forceinline__ int choose_vec(const float* origin, int32_t block_size, int* lpb_log2) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(origin);
  auto pow2 = [](int32_t x) { return x > 0 && (x & (x - 1)) == 0; };
  int vec = 0;
  if (block_size % 4 == 0 && (a & 15) == 0 && pow2(block_size / 4))
    vec = 4;
  else if (block_size % 2 == 0 && (a & 7) == 0 && pow2(block_size / 2))
    vec = 2;
  else if (pow2(block_size))
    vec = 1;
  if (vec) *lpb_log2 = __ffs(block_size / vec) - 1;
  return vec;
}

// Unsharded dispatch: vector width chosen per row at run time.
__device__ __forceinline__ void stream_row(const Window& w, int vec, int lpb_log2,
                                           int32_t block_size, int32_t b0, int32_t b1,
                                           uint32_t* keys, int32_t kbase) {
  switch (vec) {
    case 4: stream_pow2<4, 4, 1>(w, lpb_log2, b0, b1, keys, kbase); break;
    case 2: stream_pow2<2, 8, 1>(w, lpb_log2, b0, b1, keys, kbase); break;
    case 1: stream_pow2<1, 16, 1>(w, lpb_log2, b0, b1, keys, kbase); break;
    default: stream_generic<8, 1>(w, block_size, b0, b1, keys, kbase); break;
  }
}

}  // namespace dsa
