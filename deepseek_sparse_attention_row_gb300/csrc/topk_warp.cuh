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
// shared memory, 16-byte aligned. out: the row's output slots (global;
// unused when k == 0).
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
      // Candidates read in 16-byte pairs (cand is 16-byte aligned).
      const ulonglong2* pairs = reinterpret_cast<const ulonglong2*>(cand);
      for (int i = lane; i < n; i += 32) {
        const uint64_t ci = cand[i];
        int32_t r = 0;
#pragma unroll 4
        for (int j = 0; j < (n >> 1); ++j) {
          const ulonglong2 cj = pairs[j];
          r += (cj.x > ci) + (cj.y > ci);
        }
        if (n & 1) r += cand[n - 1] > ci;
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

// R-th largest of the 32 lanes' values v, counted with multiplicity, or 0
// when fewer than R lanes hold a value above key(-inf). At most R rounds of a
// warp max, each dropping the lanes that hold it. Warp-uniform result.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t v, int R) {
  for (int need = R; need > 0;) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, v);
    if (m <= kKeyNegInf) return 0u;
    const int c = __popc(__ballot_sync(0xffffffffu, v == m));
    if (c >= need) return m;
    need -= c;
    if (v == m) v = 0u;
  }
  return 0u;
}

// Ranked top-k of one row by one warp for rows of up to 1024 block keys
// (32 per lane) and k <= 32; same result as topk_store. Lane l holds keys
// l, l + 32, ... (conflict-free loads; a short row still spreads over the
// lanes) and keeps its two largest t1 >= t2. Bound: ceil(k/2) lanes with
// t2 >= L hold at least k keys >= L, so every top-k key is >= L; when fewer
// than ceil(k/2) lanes hold two live keys, every live key is a candidate.
// Candidates (typically k plus a few dozen) are marked in a 32-bit mask per
// lane, a warp scan of the mask counts gives each lane its slots, and each is
// ranked by counting the composites above it. More candidates than
// `cand_cap` (long runs of equal keys): k rounds of a warp max.
//
// keys: [n_live] final keys in shared memory (no other warp writes them any
// more); block pin_block (if >= 0, below n_live) becomes key(+inf) here.
// cand: [cand_cap >= 64, even] in shared memory, 16-byte aligned. All 32
// lanes call this.
template <typename S>
__device__ void topk_warp_wide(uint32_t* __restrict__ keys, int32_t nb, int32_t n_live, int32_t k,
                               int32_t pin_block, uint64_t* __restrict__ cand, int32_t cand_cap,
                               int32_t* __restrict__ out, int32_t topk, S* __restrict__ scores) {
  const int lane = threadIdx.x & 31;
  if (lane == 0 && pin_block >= 0) keys[pin_block] = kKeyPosInf;
  __syncwarp();
  if (scores)
    for (int b = lane; b < nb; b += 32) put_score(scores + b, b < n_live ? keys[b] : kKeyNegInf);
  if (k <= 0) return;

  // 1. Each lane's two largest keys (0 stands for none: every key is >=
  // key(-inf) > 0), over the rounds of 32 keys the row has.
  const int rounds = (n_live + 31) >> 5;
  uint32_t t1 = 0u, t2 = 0u;
#pragma unroll 8
  for (int i = 0; i < rounds; ++i) {
    const int b = lane + 32 * i;
    const uint32_t x = b < n_live ? keys[b] : 0u;
    t2 = max(t2, min(t1, x));
    t1 = max(t1, x);
  }

  // 2. The bound (key(-inf) + 1, i.e. every live key, when it fails).
  uint32_t thr = warp_kth_largest(t2, (k + 1) >> 1);
  const bool take_all = thr == 0u;
  if (take_all) thr = kKeyNegInf + 1u;

  // 3. Candidates: a bit per key at or above the bound, then a warp scan of
  // the counts gives each lane its slots.
  uint32_t bits = 0u;
#pragma unroll 8
  for (int i = 0; i < rounds; ++i) {
    const int b = lane + 32 * i;
    bits |= (b < n_live && keys[b] >= thr) ? (1u << i) : 0u;
  }
  const uint32_t mine = __popc(bits);
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int32_t n = static_cast<int32_t>(__shfl_sync(0xffffffffu, incl, 31));
  const int32_t K = take_all ? min(k, n) : k;
  if (K == 0) {
    for (int j = lane; j < topk; j += 32) out[j] = -1;
    return;
  }
  if (n <= cand_cap) {
    int32_t pos = static_cast<int32_t>(incl - mine);
    while (bits) {
      const int q = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int b = lane + 32 * q;
      cand[pos++] = pack_candidate(keys[b], b);
    }
    // An odd count is padded with a 0 composite (below every candidate), so
    // that the ranking reads pairs with 16-byte loads.
    if (lane == 0 && (n & 1)) cand[n] = 0ull;
    __syncwarp();
    // 4. Rank by counting; two candidates per lane per pass.
    const ulonglong2* pairs = reinterpret_cast<const ulonglong2*>(cand);
    for (int i0 = 0; i0 < n; i0 += 64) {
      const int ia = i0 + lane, ib = i0 + 32 + lane;
      const uint64_t ca = ia < n ? cand[ia] : 0ull;
      const uint64_t cb = ib < n ? cand[ib] : 0ull;
      int32_t ra = 0, rb = 0;
#pragma unroll 4
      for (int j = 0; j < (n + 1) >> 1; ++j) {
        const ulonglong2 cj = pairs[j];
        ra += (cj.x > ca) + (cj.y > ca);
        rb += (cj.x > cb) + (cj.y > cb);
      }
      if (ia < n && ra < K) out[ra] = candidate_id(ca);
      if (ib < n && rb < K) out[rb] = candidate_id(cb);
    }
    for (int j = K + lane; j < topk; j += 32) out[j] = -1;
    return;
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
