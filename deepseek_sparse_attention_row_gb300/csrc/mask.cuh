// mask.cuh -- masking packed logits to the selected candidate blocks.
//
// candidate_blocks.py diff, the masking function after selection ("mask
// packed logits outside causal bounds and request-local candidates"; under
// DCP the local block size is passed and the candidate ids apply unchanged).
// In place: logit c of a row becomes -inf when c is outside the row's window
// [s, e) or its request-local block (c - s) / block_size is not one of the
// row's candidate ids (ids < 0 are empty slots). Kept logits are not touched,
// so the pass never reads the logits: it only writes -inf.
//
// One CTA per (shard, row, chunk of kMaskChunk columns). The CTA first marks
// the candidate blocks overlapping its chunk in a shared-memory bitmap, then
// walks the chunk in 16-byte-aligned slots: a slot whose four columns are all
// masked gets one 16-byte store, a slot at a window or chunk edge gets scalar
// stores for its masked columns.
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

constexpr int32_t kMaskChunk = 8192;                    // columns per CTA
constexpr int32_t kMaskBitmapWords = (kMaskChunk + 64) / 32 + 1;

struct MaskArgs {
  float* logits;
  int64_t ld;
  int64_t shard_stride;
  int32_t shards;        // 1: unsharded
  int64_t rows;
  int32_t width;         // (local) width
  const int32_t* row_ks;  // unsharded only, nullable
  const int32_t* row_ke;  // unsharded: ends; sharded: global ends
  int32_t row_repeat;
  int32_t block_size;    // (local) block
  const int32_t* cand;
  int32_t topk;
  int64_t ld_cand;
  int32_t chunks;        // chunks per row
};

__device__ __forceinline__ void st_neg_inf4(float* p) {
  const float n = neg_inf();
  asm volatile("st.global.v4.f32 [%0], {%1, %1, %1, %1};" ::"l"(p), "f"(n) : "memory");
}

__global__ void __launch_bounds__(256) mask_kernel(const MaskArgs a) {
  __shared__ uint32_t bits[kMaskBitmapWords];
  const int64_t unit = blockIdx.x / a.chunks;  // shard-major: unit = d * rows + row
  const int32_t chunk = static_cast<int32_t>(blockIdx.x % a.chunks);
  const int32_t d = static_cast<int32_t>(unit / a.rows);
  const int64_t row = unit % a.rows;
  const int64_t g = row / a.row_repeat;

  // Window of this (shard, row).
  int32_t s, e;
  if (a.shards == 1) {
    const int32_t ks = a.row_ks ? __ldg(a.row_ks + g) : 0;
    const int32_t ke = __ldg(a.row_ke + g);
    e = min(ke, a.width);
    s = min(max(ks, 0), e);
  } else {
    const int32_t gke = __ldg(a.row_ke + g);
    s = 0;
    e = 0;
    if (gke > d) {
      const uint32_t lke = (static_cast<uint32_t>(gke - d) + static_cast<uint32_t>(a.shards - 1)) /
                           static_cast<uint32_t>(a.shards);
      e = static_cast<int32_t>(min(lke, static_cast<uint32_t>(a.width)));
    }
  }
  const int32_t c0 = chunk * kMaskChunk;
  const int32_t c1 = min(c0 + kMaskChunk, a.width);
  // Blocks that can hold kept columns of this chunk: [blo, bhi).
  const int32_t lo_c = max(c0, s), hi_c = min(c1, e);
  const int32_t blo = lo_c < hi_c ? (lo_c - s) / a.block_size : 0;
  const int32_t bhi = lo_c < hi_c ? (hi_c - 1 - s) / a.block_size + 1 : 0;
  const int32_t nbits = bhi - blo;  // <= kMaskChunk + 1
  for (int i = threadIdx.x; i < kMaskBitmapWords; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  if (nbits > 0) {
    const int32_t* crow = a.cand + row * a.ld_cand;
    for (int j = threadIdx.x; j < a.topk; j += blockDim.x) {
      const int32_t b = __ldg(crow + j);
      if (b >= blo && b < bhi) atomicOr(&bits[(b - blo) >> 5], 1u << ((b - blo) & 31));
    }
  }
  __syncthreads();

  float* rowp = a.logits + static_cast<int64_t>(d) * a.shard_stride + row * a.ld;
  auto kept = [&](int32_t c) -> bool {
    if (c < s || c >= e) return false;
    const int32_t b = (c - s) / a.block_size - blo;
    return (bits[b >> 5] >> (b & 31)) & 1u;
  };
  // 16-byte slots: slot k covers columns [a0 + 4k, a0 + 4k + 4).
  const int32_t mis = static_cast<int32_t>((reinterpret_cast<uintptr_t>(rowp + c0) >> 2) & 3);
  const int32_t a0 = c0 - mis;
  const int32_t nslots = (c1 - a0 + 3) / 4;
  for (int32_t k = threadIdx.x; k < nslots; k += blockDim.x) {
    const int32_t cb = a0 + 4 * k;
    const bool inside = cb >= c0 && cb + 4 <= c1;
    // Fast case: all four columns outside the window.
    if (inside && (cb + 4 <= s || cb >= e)) {
      st_neg_inf4(rowp + cb);
      continue;
    }
    bool m[4];
    bool all = inside;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int32_t c = cb + i;
      m[i] = c >= c0 && c < c1 && !kept(c);
      all = all && m[i];
    }
    if (all) {
      st_neg_inf4(rowp + cb);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (m[i]) rowp[cb + i] = neg_inf();
    }
  }
}

}  // namespace dsa
