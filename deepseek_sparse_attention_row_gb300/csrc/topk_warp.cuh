// topk_warp.cuh -- ranked top-k of one row by a single warp, with no CTA
// barrier (rows handled one per warp, see select_warp_kernel).
//
// Same result as topk_store (topk.cuh): candidates are the 64-bit composites
// (key << 32) | ~id, ranked descending, so ties rank the lower id first; a
// slot past K = min(k, keys above -inf) holds -1. k <= 32.
//
// Fast path (up to 8 live keys per lane): lane l holds keys l, l + 32, ... in
// registers. With K <= 32 the K-th largest lane max is a bound: K lanes each
// hold a key at or above it. Keys at or above the bound are compacted into
// shared memory with ballots (no atomics), and each is ranked by counting the
// candidates above it. Fallback (more live keys, or more candidates than
// kWarpCand): K rounds of a warp-wide max over the composites below the last
// one taken, reading the keys from shared memory.
#pragma once

#include <cstdint>

#include "keys.cuh"
#include "topk.cuh"

namespace dsa {

constexpr int kWarpCand = 128;  // candidates ranked by counting, per warp

// keys: this warp's [n_live] block keys in shared memory (the pinned block,
// if >= 0, lies below n_live and becomes +inf here). cand: [kWarpCand] in
// shared memory. out: the row's output slots (global; unused when k == 0).
// scores: optional row of nb entries (fp32 or bf16 bits). All 32 lanes call
// this.
template <typename S>
__device__ void topk_warp(uint32_t* __restrict__ keys, int32_t nb, int32_t n_live, int32_t k,
                          int32_t pin_block, uint64_t* __restrict__ cand,
                          int32_t* __restrict__ out, int32_t topk, S* __restrict__ scores) {
  constexpr int KR = 8;
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const bool in_regs = n_live <= 32 * KR;

  if (scores)
    for (int b = lane; b < nb; b += 32)
      put_score(scores + b, b == pin_block ? kKeyPosInf : (b < n_live ? keys[b] : kKeyNegInf));

  uint32_t kr[KR];
  uint32_t cnt = 0, mx = 0;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      const int b = lane + 32 * i;
      uint32_t key = b < n_live ? keys[b] : kKeyNegInf;
      if (b == pin_block) {
        key = kKeyPosInf;
        keys[b] = key;
      }
      kr[i] = key;
      if (key > kKeyNegInf) {
        ++cnt;
        mx = max(mx, key);
      }
    }
  } else {
    for (int b = lane; b < n_live; b += 32) {
      uint32_t key = keys[b];
      if (b == pin_block) {
        key = kKeyPosInf;
        keys[b] = key;
      }
      cnt += key > kKeyNegInf;
    }
  }
  __syncwarp();
  const uint32_t total = __reduce_add_sync(0xffffffffu, cnt);
  if (k <= 0) return;
  const int32_t K = static_cast<int32_t>(min(static_cast<uint32_t>(k), total));

  if (K > 0 && in_regs) {
    uint32_t thr = kKeyNegInf + 1u;  // every key above -inf when K == total
    if (static_cast<uint32_t>(K) < total) {
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) {
        const uint32_t o = __shfl_sync(0xffffffffu, mx, j);
        rank += (o > mx) || (o == mx && j < lane);
      }
      const uint32_t who = __ballot_sync(0xffffffffu, rank == K - 1);
      thr = max(__shfl_sync(0xffffffffu, mx, __ffs(who) - 1), kKeyNegInf + 1u);
    }
    int32_t n = 0;
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      const bool take = kr[i] >= thr;
      const uint32_t bal = __ballot_sync(0xffffffffu, take);
      const int32_t pos = n + __popc(bal & lt);
      if (take && pos < kWarpCand) cand[pos] = pack_candidate(kr[i], lane + 32 * i);
      n += __popc(bal);
    }
    __syncwarp();
    if (n <= kWarpCand) {
      for (int i = lane; i < n; i += 32) {
        const uint64_t ci = cand[i];
        int32_t r = 0;
        for (int j = 0; j < n; ++j) r += cand[j] > ci;
        if (r < K) out[r] = candidate_id(ci);
      }
      for (int j = K + lane; j < topk; j += 32) out[j] = -1;
      return;
    }
  }

  // Fallback: K rounds, each taking the largest composite below the last.
  uint64_t last = ~0ull;
  for (int32_t j = 0; j < K; ++j) {
    uint64_t best = 0ull;
    for (int b = lane; b < n_live; b += 32) {
      const uint32_t key = keys[b];
      if (key > kKeyNegInf) {
        const uint64_t c = pack_candidate(key, b);
        if (c < last && c > best) best = c;
      }
    }
    const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(best >> 32));
    const uint32_t lo = __reduce_max_sync(
        0xffffffffu, static_cast<uint32_t>(best >> 32) == hi ? static_cast<uint32_t>(best) : 0u);
    best = (static_cast<uint64_t>(hi) << 32) | lo;
    if (lane == 0) out[j] = candidate_id(best);
    last = best;
  }
  for (int j = K + lane; j < topk; j += 32) out[j] = -1;
}

}  // namespace dsa
