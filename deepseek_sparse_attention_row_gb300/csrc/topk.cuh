// topk.cuh -- ranked top-k of one row's block keys, in shared memory.
//
// candidate_blocks.py diff: after the block scores, _select_candidate_blocks_impl
// takes scores.topk(min(topk_blocks, nblocks)) and _store_candidates_kernel
// writes the ids, -1 padded. Here the whole step runs in one CTA on keys that
// never leave shared memory:
//
//  1. Count the keys above key(-inf) (a -inf block can only yield -1) and
//     take their min m and max M. K = min(k, count) survivors are needed. If
//     every such key survives there is nothing to select.
//  2. Radix select for the K-th largest key. All keys in [m, M] share the
//     bits above the highest bit where m and M differ, so the digits start
//     right below that common prefix: the first histogram already spreads
//     the keys (block maxima of similar rows share their top byte, which
//     would put every key in one bin). Each pass histograms up to 8 bits of
//     the keys that still match the prefix found so far and takes the digit
//     where the running count from the top reaches the number still needed;
//     when that digit's bin holds exactly what is still needed, every key
//     with the new prefix is in and the search stops.
//  3. Gather keys above the threshold; when the threshold key itself is
//     tied, the lowest ids among the tied keys (ties rank the lower id
//     first) are added by an ordered two-phase warp scan.
//  4. Sort the K survivors descending by (key, -id) packed in 64 bits: one
//     warp's shuffle bitonic network when K <= 32, otherwise a bitonic
//     network in shared memory. Store ids, then -1 up to topk.
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

struct TopkShared {
  uint32_t hist[2][256];
  uint32_t warp_count[32], warp_max[32], warp_min[32];
  uint32_t digit, above, eq;
  uint32_t count_gt;
};

__device__ __forceinline__ uint64_t pack_candidate(uint32_t key, int32_t id) {
  return (static_cast<uint64_t>(key) << 32) |
         static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int32_t candidate_id(uint64_t c) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
}

// keys: [nb] in shared memory (final). cand: [kpad] in shared memory, kpad a
// power of two >= min(k, nb). out: this row's output slots (global). Every
// thread of the CTA calls this.
__device__ void topk_store(const uint32_t* __restrict__ keys, int32_t nb, int32_t k,
                           uint64_t* __restrict__ cand, int32_t kpad, int32_t* __restrict__ out,
                           int32_t topk, TopkShared& sh) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int nwarps = nthreads >> 5;

  // 1. Count, min and max of the keys above -inf.
  {
    uint32_t cnt = 0, mx = 0, mn = 0xFFFFFFFFu;
    for (int b = tid; b < nb; b += nthreads) {
      const uint32_t key = keys[b];
      if (key > kKeyNegInf) {
        ++cnt;
        mx = max(mx, key);
        mn = min(mn, key);
      }
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 0) {
      sh.warp_count[warp] = cnt;
      sh.warp_max[warp] = mx;
      sh.warp_min[warp] = mn;
    }
    for (int i = tid; i < 256; i += nthreads) sh.hist[0][i] = 0;
    if (tid == 0) sh.count_gt = 0;
  }
  __syncthreads();
  uint32_t total = 0, M = 0, m = 0xFFFFFFFFu;
  for (int i = 0; i < nwarps; ++i) {
    total += sh.warp_count[i];
    M = max(M, sh.warp_max[i]);
    m = min(m, sh.warp_min[i]);
  }
  const int32_t K = static_cast<int32_t>(min(static_cast<uint32_t>(k), total));

  // 2. Threshold: selected = keys >= prefix (take_all) or keys > prefix plus
  // `need` tied keys equal to prefix.
  uint32_t prefix = kKeyNegInf + 1u;
  bool take_all = true;
  int32_t need = 0;
  if (K > 0 && static_cast<uint32_t>(K) < total) {
    const uint32_t diff = m ^ M;
    take_all = false;
    need = K;
    if (diff == 0) {
      prefix = M;  // every candidate key is equal: all ties
    } else {
      const int hb = 31 - __clz(diff);
      uint32_t mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);
      prefix = M & mask;
      int hi = hb;
      int pass = 0;
      while (hi >= 0) {
        const int lo = max(hi - 7, 0);
        const uint32_t width_mask = (2u << (hi - lo)) - 1u;
        uint32_t* hcur = sh.hist[pass & 1];
        uint32_t* hnext = sh.hist[(pass + 1) & 1];
        for (int b = tid; b < nb; b += nthreads) {
          const uint32_t key = keys[b];
          if (key > kKeyNegInf && (key & mask) == prefix) atomicAdd(&hcur[(key >> lo) & width_mask], 1u);
        }
        for (int i = tid; i < 256; i += nthreads) hnext[i] = 0;
        __syncthreads();
        if (warp == 0) {
          // Lane l owns digits 255 - 8l down to 248 - 8l (highest first).
          uint32_t c[8], sum = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            c[i] = hcur[255 - 8 * lane - i];
            sum += c[i];
          }
          uint32_t incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const uint32_t hit = __ballot_sync(0xffffffffu, incl >= static_cast<uint32_t>(need));
          if (lane == __ffs(hit) - 1) {
            uint32_t run = incl - sum;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (run + c[i] >= static_cast<uint32_t>(need)) {
                sh.digit = 255u - 8u * lane - i;
                sh.above = run;
                sh.eq = c[i];
                break;
              }
              run += c[i];
            }
          }
        }
        __syncthreads();
        prefix |= sh.digit << lo;
        mask |= width_mask << lo;
        need -= static_cast<int32_t>(sh.above);
        if (static_cast<uint32_t>(need) == sh.eq) {
          take_all = true;
          need = 0;
          break;
        }
        hi = lo - 1;
        ++pass;
      }
    }
  }

  // 3. Gather.
  if (K > 0) {
    for (int b = tid; b < nb; b += nthreads) {
      const uint32_t key = keys[b];
      const bool sel = take_all ? (key >= prefix && key > kKeyNegInf) : (key > prefix);
      if (sel) cand[atomicAdd(&sh.count_gt, 1u)] = pack_candidate(key, b);
    }
  }
  if (need > 0) {
    // Ordered tie pass: warp w scans ids [w*span, (w+1)*span) in order.
    const int32_t span = ((nb + nwarps - 1) / nwarps + 31) & ~31;
    const int32_t lo_id = warp * span, hi_id = min(lo_id + span, nb);
    uint32_t mine = 0;
    for (int32_t base = lo_id; base < hi_id; base += 32) {
      const int32_t b = base + lane;
      mine += __popc(__ballot_sync(0xffffffffu, b < hi_id && keys[b] == prefix));
    }
    if (lane == 0) sh.warp_count[warp] = mine;
    __syncthreads();
    int32_t rank0 = 0;
    for (int i = 0; i < warp; ++i) rank0 += static_cast<int32_t>(sh.warp_count[i]);
    const int32_t count_gt = static_cast<int32_t>(sh.count_gt);
    for (int32_t base = lo_id; base < hi_id && rank0 < need; base += 32) {
      const int32_t b = base + lane;
      const bool tie = b < hi_id && keys[b] == prefix;
      const uint32_t bal = __ballot_sync(0xffffffffu, tie);
      const int32_t rank = rank0 + __popc(bal & ((1u << lane) - 1u));
      if (tie && rank < need) cand[count_gt + rank] = pack_candidate(prefix, b);
      rank0 += __popc(bal);
    }
  }
  __syncthreads();

  // 4. Sort survivors descending and store.
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
          v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
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
