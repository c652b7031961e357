// topk.cuh -- ranked top-k of one row's block keys, in shared memory.
//
// candidate_blocks.py diff: after the block scores, _select_candidate_blocks_impl
// takes scores.topk(min(topk_blocks, nblocks)) and _store_candidates_kernel
// writes the ids, -1 padded. Here the whole step runs in one CTA on keys that
// never leave shared memory:
//
//  1. Radix select on the 32-bit order keys, most significant byte first,
//     over the keys above key(-inf) (a -inf block can only ever yield -1):
//     each pass histograms one byte of the keys that still match the prefix
//     found so far and picks the byte value where the running count from the
//     top reaches the number still needed. If that byte's bin holds exactly
//     what is still needed, every key with the prefix is in and the search
//     stops early.
//  2. Gather: keys strictly above the threshold go straight in; when the
//     threshold key itself is tied, the lowest ids among the tied keys are
//     taken with an ordered block-wide scan (ties rank the lower id first).
//  3. Sort the K <= k survivors descending by (key, -id) packed in 64 bits:
//     one warp's shuffle bitonic network when K <= 32, otherwise a bitonic
//     network in shared memory.
//  4. Store ids, then -1 for every remaining slot up to topk.
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

struct TopkShared {
  uint32_t hist[256];
  uint32_t digit, above, eq, total;
  uint32_t count_gt;
  uint32_t warp_count[32];
};

__device__ __forceinline__ uint64_t pack_candidate(uint32_t key, int32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int32_t candidate_id(uint64_t c) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
}

// keys: [nb] in shared memory. cand: [kpad] in shared memory, kpad a power of
// two >= min(k, nb). out: this row's output slots (global). Called by every
// thread of the CTA.
__device__ void topk_store(const uint32_t* __restrict__ keys, int32_t nb, int32_t k,
                           uint64_t* __restrict__ cand, int32_t kpad, int32_t* __restrict__ out,
                           int32_t topk, TopkShared& sh) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nthreads = blockDim.x;

  uint32_t prefix = 0, mask = 0;
  int32_t need = 0;       // survivors still to choose at the current prefix
  int32_t total_k = 0;    // K: survivors in all
  bool take_all_with_prefix = false;

  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += nthreads) sh.hist[i] = 0;
    __syncthreads();
    for (int b = tid; b < nb; b += nthreads) {
      const uint32_t key = keys[b];
      if (key > kKeyNegInf && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // Lane l owns digits 255 - 8l down to 248 - 8l (highest first).
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = sh.hist[255 - 8 * lane - i];
        sum += c[i];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t want = (pass == 0) ? min(static_cast<uint32_t>(k), total) : static_cast<uint32_t>(need);
      if (pass == 0 && lane == 0) sh.total = total;
      if (want > 0) {
        const uint32_t hit = __ballot_sync(0xffffffffu, incl >= want);
        const int first = __ffs(hit) - 1;
        if (lane == first) {
          uint32_t run = incl - sum;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run + c[i] >= want) {
              sh.digit = 255u - 8u * lane - i;
              sh.above = run;
              sh.eq = c[i];
              break;
            }
            run += c[i];
          }
        }
      }
    }
    __syncthreads();
    if (pass == 0) {
      const uint32_t total = sh.total;
      total_k = static_cast<int32_t>(min(static_cast<uint32_t>(k), total));
      if (total_k == 0) break;
      if (static_cast<uint32_t>(total_k) == total) {
        // Every key above -inf is a survivor.
        prefix = kKeyNegInf + 1u;
        take_all_with_prefix = true;
        need = 0;
        break;
      }
      need = total_k;
    }
    prefix |= sh.digit << shift;
    mask |= 255u << shift;
    need -= static_cast<int32_t>(sh.above);
    if (static_cast<uint32_t>(need) == sh.eq) {
      take_all_with_prefix = true;
      need = 0;
      break;
    }
  }

  // Gather survivors.
  if (tid == 0) sh.count_gt = 0;
  __syncthreads();
  if (total_k > 0) {
    for (int b = tid; b < nb; b += nthreads) {
      const uint32_t key = keys[b];
      const bool sel = take_all_with_prefix ? (key >= prefix && key > kKeyNegInf) : (key > prefix);
      if (sel) cand[atomicAdd(&sh.count_gt, 1u)] = pack_candidate(key, b);
    }
  }
  __syncthreads();
  const int32_t count_gt = static_cast<int32_t>(sh.count_gt);
  if (!take_all_with_prefix && need > 0) {
    // prefix is the full threshold key; take the `need` lowest tied ids.
    int32_t taken = 0;
    const int nw = nthreads >> 5;
    for (int base = 0; base < nb && taken < need; base += nthreads) {
      const int b = base + tid;
      const bool tie = b < nb && keys[b] == prefix;
      const uint32_t bal = __ballot_sync(0xffffffffu, tie);
      if (lane == 0) sh.warp_count[warp] = __popc(bal);
      __syncthreads();
      int32_t before = 0, tile = 0;
      for (int i = 0; i < nw; ++i) {
        const int32_t c = static_cast<int32_t>(sh.warp_count[i]);
        before += (i < warp) ? c : 0;
        tile += c;
      }
      const int32_t rank = taken + before + __popc(bal & ((1u << lane) - 1u));
      if (tie && rank < need) cand[count_gt + rank] = pack_candidate(prefix, b);
      taken += tile;
      __syncthreads();
    }
  }
  const int32_t K = total_k;
  __syncthreads();

  // Sort survivors descending and store.
  if (kpad <= 32) {
    if (warp == 0) {
      uint64_t v = (lane < K) ? cand[lane] : 0ull;
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
          const bool desc = (lane & size) == 0;
          const bool lower = (lane & stride) == 0;
          const bool keep_max = (lower == desc);
          v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
        }
      }
      if (lane < topk) out[lane] = (lane < K) ? candidate_id(v) : -1;
    }
    for (int j = 32 + tid; j < topk; j += nthreads) out[j] = -1;
    return;
  }
  for (int i = K + tid; i < kpad; i += nthreads) cand[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= kpad; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (kpad >> 1); i += nthreads) {
        const int lo = ((i / stride) * stride * 2) + (i % stride);
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = cand[lo], b = cand[hi];
        if ((a < b) == desc) {
          cand[lo] = b;
          cand[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = tid; j < topk; j += nthreads) out[j] = (j < K) ? candidate_id(cand[j]) : -1;
}

}  // namespace dsa
