// topk.cuh -- ranked top-k of one row's block keys, in shared memory.
//
// candidate_blocks.py diff: after the block scores, _select_candidate_blocks_impl
// takes scores.topk(min(topk_blocks, nblocks)) and _store_candidates_kernel
// writes the ids, -1 padded. Here the whole step runs in one CTA on keys that
// never leave shared memory. Every candidate is the 64-bit composite
// (key << 32) | ~id, so composites are distinct and their descending order is
// exactly "score descending, then lower id first". Only keys above key(-inf)
// can be selected (a -inf block yields -1); K = min(k, their count).
//
// Only the row's live blocks are touched: blocks past the last one holding
// in-window data (or the pin) are -inf by construction.
//
// Fast path (k <= 32 * warps, up to 8 live keys per thread): thread t holds
// keys t, t + T, ... in registers. Each warp ranks its 32 lane maxima with
// shuffles and takes the R-th largest, R = ceil(k / warps): R lanes each hold
// a key at or above it, so every warp has at least R keys >= its value and
// at least k keys are >= L, the smallest of the warps' values. The
// candidates are the keys >= L (a few more than k on typical rows); each is
// ranked by counting the candidates above it and rank r < K is stored in
// slot r. Two barriers, no sort network, no tie handling.
//
// Exact path (larger k, or more candidates than kRankMax): radix select for
// the K-th largest key with 8-bit digits starting right below the common
// prefix of the row's min and max key; the lowest tied ids at the threshold
// are taken by an ordered warp scan; the K survivors are then ranked by
// counting (K <= kRankMax) or sorted by a bitonic network in shared memory.
#pragma once

#include <cstdint>

#include "keys.cuh"

namespace dsa {

constexpr int kRankMax = 256;  // candidates ranked by counting

// Which threads take part in a row's top-k, and how they meet. CtaSync: every
// thread of the CTA, __syncthreads(). NamedSync<N, ID, BASE>: the N threads
// BASE .. BASE + N - 1 (whole warps), named barrier ID, so that the CTA's
// other warps (a producer, the warps folding the next row) carry on
// meanwhile. tid() is a thread's index within the group.
struct CtaSync {
  __device__ __forceinline__ static void sync() { __syncthreads(); }
  __device__ __forceinline__ static int count() { return blockDim.x; }
  __device__ __forceinline__ static int tid() { return threadIdx.x; }
};
template <int N, int ID = 1, int BASE = 0>
struct NamedSync {
  static_assert(N % 32 == 0 && BASE % 32 == 0, "whole warps");
  __device__ __forceinline__ static void sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
  }
  __device__ __forceinline__ static constexpr int count() { return N; }
  __device__ __forceinline__ static int tid() { return static_cast<int>(threadIdx.x) - BASE; }
};

struct TopkShared {
  uint32_t hist[256];
  uint32_t warp_count[32], warp_kth[32], warp_max[32], warp_min[32];
  uint32_t digit, above, eq;
  uint32_t count;
};

__device__ __forceinline__ uint64_t pack_candidate(uint32_t key, int32_t id) {
  return (static_cast<uint64_t>(key) << 32) |
         static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int32_t candidate_id(uint64_t c) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
}

// Stores ranks of cand[0 .. n) (distinct composites): rank r < K goes to
// out[r]; out[K .. topk) becomes -1. No barrier inside.
// cand is 16-byte aligned: the candidates are read in pairs.
template <typename Sync = CtaSync>
__device__ __forceinline__ void rank_store(const uint64_t* __restrict__ cand, int32_t n, int32_t K,
                                           int32_t* __restrict__ out, int32_t topk) {
  const ulonglong2* pairs = reinterpret_cast<const ulonglong2*>(cand);
  for (int i = Sync::tid(); i < n; i += Sync::count()) {
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
  for (int j = K + Sync::tid(); j < topk; j += Sync::count()) out[j] = -1;
}

// Exact path. Preconditions: keys final; total = number of keys above -inf,
// m / M their min / max, 0 < K <= total. Ends with the row stored.
template <typename Sync = CtaSync>
__device__ void topk_exact(const uint32_t* __restrict__ keys, int32_t nb, int32_t K, uint32_t total,
                           uint32_t m, uint32_t M, uint64_t* __restrict__ cand, int32_t kpad,
                           int32_t* __restrict__ out, int32_t topk, TopkShared& sh) {
  const int tid = Sync::tid();
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nthreads = Sync::count();
  const int nwarps = nthreads >> 5;

  if (tid == 0) sh.count = 0;
  for (int i = tid; i < 256; i += nthreads) sh.hist[i] = 0;
  Sync::sync();

  uint32_t prefix = kKeyNegInf + 1u;  // selected: keys >= prefix (take_all) or
  bool take_all = true;               // keys > prefix plus `need` tied keys
  int32_t need = 0;
  if (static_cast<uint32_t>(K) < total) {
    take_all = false;
    need = K;
    if (m == M) {
      prefix = M;  // every key above -inf is equal: pure ties
    } else {
      const int hb = 31 - __clz(m ^ M);
      uint32_t mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);
      prefix = M & mask;
      int hi = hb;
      for (int pass = 0; hi >= 0; ++pass) {
        const int lo = max(hi - 7, 0);
        const uint32_t wmask = (2u << (hi - lo)) - 1u;
        if (pass > 0) {
          for (int i = tid; i < 256; i += nthreads) sh.hist[i] = 0;
          Sync::sync();
        }
        for (int b = tid; b < nb; b += nthreads) {
          const uint32_t key = keys[b];
          if (key > kKeyNegInf && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> lo) & wmask], 1u);
        }
        Sync::sync();
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
        Sync::sync();
        prefix |= sh.digit << lo;
        mask |= wmask << lo;
        need -= static_cast<int32_t>(sh.above);
        if (static_cast<uint32_t>(need) == sh.eq) {
          take_all = true;
          need = 0;
          break;
        }
        hi = lo - 1;
      }
    }
  }

  // Gather exactly K survivors.
  for (int b = tid; b < nb; b += nthreads) {
    const uint32_t key = keys[b];
    const bool sel = take_all ? (key >= prefix && key > kKeyNegInf) : (key > prefix);
    if (sel) cand[atomicAdd(&sh.count, 1u)] = pack_candidate(key, b);
  }
  if (need > 0) {
    // Ordered tie pass: warp w scans ids [w*span, (w+1)*span) in order and
    // the lowest `need` tied ids overall are taken.
    const int32_t span = ((nb + nwarps - 1) / nwarps + 31) & ~31;
    const int32_t lo_id = warp * span, hi_id = min(lo_id + span, nb);
    uint32_t mine = 0;
    for (int32_t base = lo_id; base < hi_id; base += 32) {
      const int32_t b = base + lane;
      mine += __popc(__ballot_sync(0xffffffffu, b < hi_id && keys[b] == prefix));
    }
    if (lane == 0) sh.warp_count[warp] = mine;
    Sync::sync();
    int32_t rank0 = 0;
    for (int i = 0; i < warp; ++i) rank0 += static_cast<int32_t>(sh.warp_count[i]);
    const int32_t count_gt = static_cast<int32_t>(sh.count);
    for (int32_t base = lo_id; base < hi_id && rank0 < need; base += 32) {
      const int32_t b = base + lane;
      const bool tie = b < hi_id && keys[b] == prefix;
      const uint32_t bal = __ballot_sync(0xffffffffu, tie);
      const int32_t rank = rank0 + __popc(bal & ((1u << lane) - 1u));
      if (tie && rank < need) cand[count_gt + rank] = pack_candidate(prefix, b);
      rank0 += __popc(bal);
    }
  }
  Sync::sync();

  if (K <= kRankMax) {
    rank_store<Sync>(cand, K, K, out, topk);
    return;
  }
  for (int i = K + tid; i < kpad; i += nthreads) cand[i] = 0ull;
  Sync::sync();
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
      Sync::sync();
    }
  }
  for (int j = tid; j < topk; j += nthreads) out[j] = (j < K) ? candidate_id(cand[j]) : -1;
}

// keys: [nb] in shared memory, every block at or past n_live equal to
// key(-inf) (n_live covers the pinned block); block pin_block (if >= 0)
// becomes +inf here. cand: [max(kpad, kRankMax)] in shared memory, kpad a
// power of two >= min(k, nb). out: this row's output slots (global; unused
// when k == 0). scores: optional row (nb entries, fp32 or bf16 bits like the
// logits) written with the final scores. Every thread of the CTA calls this.
template <typename S, typename Sync = CtaSync>
__device__ void topk_store(uint32_t* __restrict__ keys, int32_t nb, int32_t n_live, int32_t k,
                           int32_t pin_block, uint64_t* __restrict__ cand, int32_t kpad,
                           int32_t* __restrict__ out, int32_t topk, S* __restrict__ scores,
                           TopkShared& sh) {
  constexpr int KR = 8;  // live keys per thread held in registers
  const int tid = Sync::tid();
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nthreads = Sync::count();
  const int nwarps = nthreads >> 5;
  const bool in_regs = n_live <= KR * nthreads;
  const bool fast = k > 0 && k <= 32 * nwarps && in_regs;
  const int R = fast ? (k + nwarps - 1) / nwarps : 0;

  if (scores)
    for (int b = tid; b < nb; b += nthreads)
      put_score(scores + b, b == pin_block ? kKeyPosInf : (b < n_live ? keys[b] : kKeyNegInf));

  // 1. Each thread takes its own keys b = tid + i*T: pin, count, min, max and
  // its largest key (lane max).
  uint32_t kr[KR];
  uint32_t cnt = 0, mx = 0, mn = 0xFFFFFFFFu;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      const int b = tid + i * nthreads;
      uint32_t key = b < n_live ? keys[b] : kKeyNegInf;
      if (b == pin_block) {
        key = kKeyPosInf;
        keys[b] = key;
      }
      kr[i] = key;
      if (key > kKeyNegInf) {
        ++cnt;
        mx = max(mx, key);
        mn = min(mn, key);
      }
    }
  } else {
    for (int b = tid; b < n_live; b += nthreads) {
      uint32_t key = keys[b];
      if (b == pin_block) {
        key = kKeyPosInf;
        keys[b] = key;
      }
      if (key > kKeyNegInf) {
        ++cnt;
        mx = max(mx, key);
        mn = min(mn, key);
      }
    }
  }
  // Warp bound: the R-th largest lane max. R lanes each hold a key at or
  // above it, so at least R of the warp's keys are >= it.
  uint32_t kth = kKeyNegInf;
  if (fast) {
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const uint32_t o = __shfl_sync(0xffffffffu, mx, j);
      rank += (o > mx) || (o == mx && j < lane);
    }
    const uint32_t who = __ballot_sync(0xffffffffu, rank == R - 1);
    kth = __shfl_sync(0xffffffffu, mx, __ffs(who) - 1);
    if (kth <= kKeyNegInf) kth = kKeyNegInf;  // fewer than R lanes hold keys
  }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  const uint32_t wmax = __reduce_max_sync(0xffffffffu, mx);
  const uint32_t wmin = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) {
    sh.warp_count[warp] = cnt;
    sh.warp_max[warp] = wmax;
    sh.warp_min[warp] = wmin;
    sh.warp_kth[warp] = kth;
  }
  if (tid == 0) sh.count = 0;
  Sync::sync();
  if (k <= 0) return;

  uint32_t total = 0, M = 0, m = 0xFFFFFFFFu, L = 0xFFFFFFFFu;
  for (int i = 0; i < nwarps; ++i) {
    total += sh.warp_count[i];
    M = max(M, sh.warp_max[i]);
    m = min(m, sh.warp_min[i]);
    L = min(L, sh.warp_kth[i]);
  }
  const int32_t K = static_cast<int32_t>(min(static_cast<uint32_t>(k), total));
  if (K == 0) {
    for (int j = tid; j < topk; j += nthreads) out[j] = -1;
    return;
  }

  if (fast) {
    // 2. Candidates: keys >= L (every key above -inf when K == total).
    const uint32_t thr = (static_cast<uint32_t>(K) == total) ? kKeyNegInf + 1u : max(L, kKeyNegInf + 1u);
    const uint32_t cap = static_cast<uint32_t>(max(kpad, kRankMax));
    // One shared atomic per warp: ballots count the warp's candidates, lane 0
    // reserves their slots, each lane writes at its prefix.
    uint32_t bal[KR], wn = 0;
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      bal[i] = __ballot_sync(0xffffffffu, kr[i] >= thr);
      wn += __popc(bal[i]);
    }
    uint32_t base = 0;
    if (lane == 0 && wn) base = atomicAdd(&sh.count, wn);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      const uint32_t pos = base + __popc(bal[i] & lt);
      if (((bal[i] >> lane) & 1u) && pos < cap) cand[pos] = pack_candidate(kr[i], tid + i * nthreads);
      base += __popc(bal[i]);
    }
    Sync::sync();
    const uint32_t n = sh.count;
    if (n <= static_cast<uint32_t>(kRankMax)) {
      // 3. Rank by counting.
      rank_store<Sync>(cand, static_cast<int32_t>(n), K, out, topk);
      return;
    }
    Sync::sync();  // every thread has read sh.count before it is reset
  }
  topk_exact<Sync>(keys, n_live, K, total, m, M, cand, kpad, out, topk, sh);
}

}  // namespace dsa
