// select_pipe.cu -- pipelined candidate-block selection: persistent CTAs that
// stage in-window logits into a shared-memory ring with the bulk-copy engine
// (cp.async.bulk, pipe.cuh) while their consumer warps reduce the previous
// stages and rank finished rows.
//
// What is computed is that of select_kernel (dsa_cb.cu) and of
// candidate_blocks.py's _block_scores_kernel, _select_candidate_blocks_impl
// and _store_candidates_kernel: per row the window [s, e) cut into blocks of
// block_size counted from s, each block's NaN-propagating max (-inf when
// empty), the optional pin, the ranked top-k with ties to the lower id, -1
// padded; in the DCP form the max over the shards' local blocks, the global
// pin and the rows without context. Only the way the bytes move differs.
//
// Layout of a CTA: warps 0 .. NW-1 consume, warp NW produces. The producer
// takes work units (a row, or a part of a long row), plans each unit's
// window from the row's bounds and cuts it into stages of whole blocks. A
// stage holds, for every shard of the row (one piece when unsharded), the
// piece of that shard's window that covers the stage's blocks, copied with
// one cp.async.bulk from the 16-byte aligned address at or below the
// piece's first element to the one at or above its end. The granules read
// beyond the piece hold at least one in-window element each, so no byte is
// read from a 16-byte granule (or page) that the window does not touch; the
// consumers never look at the extra elements. The stage's descriptor (the
// row, the block range, where each piece's first element landed and how
// many elements it has) is written before the stage's "full" barrier is
// armed with the bytes in flight.
//
// Consumers read a stage's elements from shared memory with consecutive
// lanes on consecutive elements (no bank conflicts whatever the window's
// alignment), fold the pieces with max.NaN, reduce each block across lanes
// as order keys (keys.cuh) and store the block's key once: a stage holds
// whole blocks, so no key is written twice and none needs an atomic.
//
//  - coop (all warps on one row): every consumer warp takes a share of every
//    stage's blocks; when a unit's last stage is in, the warps rank the row
//    together (topk.cuh with a named barrier, so the producer keeps
//    filling the ring meanwhile). A long row cut into parts meets in the
//    workspace as in select_kernel: each part publishes its keys, counts
//    itself in, and the last part to arrive ranks the row.
//  - solo (one row per warp): each consumer warp owns a sub-ring; the
//    producer hands whole rows to the warps in turn and each warp ranks its
//    own rows with topk_warp, without any CTA barrier.
//
// Work units: rows * S of them, unit u being part u % S of row u / S. With
// a workspace the producer takes units from a queue counter in the
// workspace (the last CTA to finish resets it to zero); without one, CTA b
// takes units b, b + grid, ... and S is 1.
#include "select_pipe.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "keys.cuh"
#include "pipe.cuh"
#include "topk.cuh"
#include "topk_warp.cuh"

namespace dsa {
namespace {

constexpr int kMaxShardLanes = 32;  // shards per row: one producer lane each
constexpr int kPipeMaxBlocks = 4096;
constexpr int kPipeMaxTopk = 256;
constexpr int32_t kPartUnit = 32;  // blocks: a part of a split row is a multiple

// Stage flags.
constexpr int32_t kLast = 2;   // last stage of a unit: rank or merge after it
constexpr int32_t kDone = 4;   // no more units for this consumer

// Wait sites recorded in g_pipe_error on a timeout.
constexpr unsigned kSiteFull = 1u, kSiteEmpty = 2u, kSiteKeys = 3u;

struct StageDesc {
  int32_t row;
  int32_t c0;       // first block of the stage (row-relative)
  int32_t n;        // blocks in the stage
  int32_t flags;
  int32_t npieces;
  int32_t nblk;     // blocks of the row holding data
  int32_t pin;      // pinned block, or -1
  int32_t b0, b1;   // the unit's blocks
  int32_t parts;    // parts of the row (1: the unit is the whole row)
  uint32_t off;     // byte offset in the stage of the piece's first element
  int32_t cnt;      // elements of the piece
};

struct PipeArgs {
  const void* logits;
  int64_t ld;
  int64_t shard_stride;
  int32_t shards;
  int32_t width;
  const int32_t* row_ks;
  const int32_t* row_ke;
  int32_t row_repeat;
  int32_t block_size;
  int32_t bs_log2;  // log2(block_size) when block_size < 32
  int32_t global_block_size;
  int32_t nb;
  int32_t nb_data;
  int32_t pin_newest;
  int32_t topk;
  int32_t kpad;
  int32_t* out;
  int64_t ld_out;
  void* scores;
  int64_t ld_scores;
  int32_t rows;
  int32_t split;        // S
  uint32_t* queue;      // [0]: next unit, [1]: CTAs done; null: static schedule
  uint32_t* ws_count;   // [rows] arrival counters (S > 1)
  uint32_t* ws_keys;    // [rows, nb] (S > 1)
  int32_t stages;       // ring depth (coop) or depth of each warp's ring (solo)
  int32_t stage_bytes;  // multiple of 128
  int32_t cap;          // blocks per stage
  int32_t own_stages;   // coop: each fold warp folds whole stages in turn
  int32_t lpt;          // coop, unsharded, S = 1: unit u is row order[u], longest first
  int32_t claim_ahead;  // coop: units claimed two ahead from the start (not as CTAs free up)
  int32_t rank_warp;    // coop: one rank warp ranks rows of <= 1024 blocks, k <= 32
};

// ---------------------------------------------------------------------------
// Shared-memory element loads
// ---------------------------------------------------------------------------

// Element of a stage, widened to fp32. `p` points into the CTA's shared
// memory (derived from the kernel's shared array, so the compiler emits
// shared loads and may batch them).
template <typename E>
__device__ __forceinline__ float stage_elem(const unsigned char* p) {
  if constexpr (E::kBytes == 4) {
    return *reinterpret_cast<const float*>(p);
  } else {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
}

// ---------------------------------------------------------------------------
// Row plans (producer side)
// ---------------------------------------------------------------------------

__device__ __forceinline__ int32_t shard_cols(int32_t gke, int32_t d, int32_t shards, int32_t lw) {
  if (gke <= d) return 0;
  const uint32_t lke = (static_cast<uint32_t>(gke - d) + static_cast<uint32_t>(shards - 1)) /
                       static_cast<uint32_t>(shards);
  return static_cast<int32_t>(min(lke, static_cast<uint32_t>(lw)));
}

// One row's plan as the producer warp holds it: lane d < shards knows shard
// d's window (first element and length); every lane knows the row totals.
template <typename E>
struct LanePlan {
  const typename E::T* origin;  // shard `lane`'s first in-window element
  int32_t len;                  // its window length (0 for lanes >= shards)
  int32_t nblk;                 // the row's blocks holding data
  int32_t pin;                  // pinned block or -1
};

// A row's bounds as read from memory: (ks or 0, ke) unsharded, (0, gke) in
// the DCP form, (gks, gke) in the DCP form with starts.
struct Bounds {
  int32_t lo, hi;
};

template <int MODE>
__device__ __forceinline__ Bounds load_bounds(const PipeArgs& a, int32_t row) {
  const int32_t g = row / a.row_repeat;
  Bounds b;
  b.lo = (MODE != kPipeSharded && a.row_ks) ? __ldg(a.row_ks + g) : 0;
  b.hi = __ldg(a.row_ke + g);
  return b;
}

template <typename E, int MODE>
__device__ __forceinline__ LanePlan<E> plan_lane(const PipeArgs& a, int32_t row, Bounds bnd,
                                                 int lane) {
  using TE = typename E::T;
  const TE* logits = static_cast<const TE*>(a.logits);
  LanePlan<E> p;
  if constexpr (MODE == kPipeUnsharded) {
    const int32_t ks = bnd.lo;
    const int32_t ke = bnd.hi;
    const int32_t e = min(ke, a.width);
    const int32_t s = min(max(ks, 0), e);
    const int32_t n = e > s ? e - s : 0;
    p.origin = logits + static_cast<int64_t>(row) * a.ld + s;
    p.len = lane == 0 ? n : 0;
    p.nblk = static_cast<int32_t>((static_cast<uint32_t>(n) + a.block_size - 1u) /
                                  static_cast<uint32_t>(a.block_size));
    p.pin = (a.pin_newest && n > 0) ? (n - 1) / a.block_size : -1;
  } else if constexpr (MODE == kPipeSharded) {
    const int32_t gke = bnd.hi;
    const int32_t n0 = shard_cols(gke, 0, a.shards, a.width);
    p.origin = logits + static_cast<int64_t>(min(lane, a.shards - 1)) * a.shard_stride +
               static_cast<int64_t>(row) * a.ld;
    p.len = lane < a.shards ? shard_cols(gke, lane, a.shards, a.width) : 0;
    p.nblk = min(static_cast<int32_t>((static_cast<uint32_t>(n0) + a.block_size - 1u) /
                                      static_cast<uint32_t>(a.block_size)),
                 a.nb_data);
    p.pin = gke >= 1 ? static_cast<int32_t>(min(static_cast<uint32_t>(gke - 1) /
                                                    static_cast<uint32_t>(a.global_block_size),
                                                static_cast<uint32_t>(a.nb - 1)))
                     : -1;
  } else {
    const int32_t gke = bnd.hi;
    const int32_t gs = min(max(bnd.lo, 0), max(gke, 0));
    const int32_t d = min(lane, a.shards - 1);
    const int32_t e = shard_cols(gke, d, a.shards, a.width);
    const int32_t st = min(shard_cols(gs, d, a.shards, a.width), e);
    p.origin = logits + static_cast<int64_t>(d) * a.shard_stride +
               static_cast<int64_t>(row) * a.ld + st;
    p.len = lane < a.shards ? e - st : 0;
    const int32_t lmax = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(p.len));
    p.nblk = min(static_cast<int32_t>((static_cast<uint32_t>(lmax) + a.block_size - 1u) /
                                      static_cast<uint32_t>(a.block_size)),
                 a.nb_data);
    p.pin = gke > gs ? static_cast<int32_t>(min(static_cast<uint32_t>(gke - gs - 1) /
                                                    static_cast<uint32_t>(a.global_block_size),
                                                static_cast<uint32_t>(a.nb - 1)))
                     : -1;
  }
  return p;
}

// The pieces of one row as the producer's lane 0 reads them, one per shard
// (one in all for unsharded rows): written by the producer warp's lanes
// (lane d: shard d) once per row.
struct PieceTable {
  const unsigned char* origin[kMaxShardLanes];  // first in-window element
  int32_t len[kMaxShardLanes];                  // window length (elements)
};

// Emits the stages of blocks [b0, b1) of one row into the ring, one piece per
// stage, in the order chunk by chunk, shard by shard within a chunk (a shard
// form's consumers merge the shards into the keys). Lane 0 alone does the
// work, so that no shuffle or warp barrier lengthens the path between two
// stages: wait for the stage's slot, write its descriptor (the unit's fields
// only on its last stage), arm its barrier and issue the one bulk copy.
// With `claim`, the next unit is claimed from the unit counter as the last
// stage's turn comes (before waiting for its slot); the counter hands out
// units from gridDim.x on (CTA b starts with unit b). Returns false (on lane
// 0) when a wait gave up.
template <typename E>
__device__ __forceinline__ bool emit_unit(const PipeArgs& a, const PieceTable& pt, int npieces,
                                          int32_t row, int32_t nblk, int32_t pin, int32_t b0,
                                          int32_t b1, int32_t parts, unsigned char* buf,
                                          uint64_t* full, uint64_t* empty, StageDesc* desc,
                                          int stages, uint32_t& k, uint32_t* claim = nullptr) {
  const int32_t bs = a.block_size;
  int32_t c = b0;
  int shard = 0;
  for (;;) {
    const int32_t n = min(a.cap, b1 - c);
    const bool last = c + n >= b1 && shard == npieces - 1;
    const uint32_t slot = k % static_cast<uint32_t>(stages);
    const uint32_t round = k / static_cast<uint32_t>(stages);
    if (last && claim) *claim = gridDim.x + atomicAdd(a.queue, 1u);
    if (round > 0 && !mbar_wait(&empty[slot], (round - 1u) & 1u, kSiteEmpty)) return false;
    // The piece: elements [c*bs, min((c+n)*bs, len)) of the shard's window,
    // copied from the 16-byte granule holding its first element through the
    // one holding its last.
    const int32_t j0 = c * bs;
    const int32_t j1 = min((c + n) * bs, pt.len[shard]);
    StageDesc& d = desc[slot];
    d.c0 = c;
    d.n = n;
    d.flags = last ? kLast : 0;
    if (last) {
      d.row = row;
      d.nblk = nblk;
      d.pin = pin;
      d.b0 = b0;
      d.b1 = b1;
      d.parts = parts;
    }
    if (j1 > j0) {
      const uintptr_t lo = reinterpret_cast<uintptr_t>(pt.origin[shard] + j0 * E::kBytes);
      const uintptr_t hi = reinterpret_cast<uintptr_t>(pt.origin[shard] + j1 * E::kBytes);
      const uintptr_t A = lo & ~static_cast<uintptr_t>(15);
      const uint32_t bytes = static_cast<uint32_t>(((hi + 15) & ~static_cast<uintptr_t>(15)) - A);
      d.off = static_cast<uint32_t>(lo - A);
      d.cnt = j1 - j0;
      mbar_arrive_expect_tx(&full[slot], bytes);
      bulk_load(buf + static_cast<size_t>(slot) * a.stage_bytes, reinterpret_cast<const void*>(A),
                bytes, &full[slot]);
    } else {
      d.off = 0;
      d.cnt = 0;
      mbar_arrive(&full[slot]);
    }
    ++k;
    if (last) return true;
    if (shard + 1 < npieces) {
      ++shard;
    } else {
      shard = 0;
      c += n;
    }
  }
}

// A stage with no data that tells its consumer(s) to stop (lane 0).
__device__ __forceinline__ bool emit_done(uint64_t* full, uint64_t* empty, StageDesc* desc,
                                          int stages, uint32_t& k) {
  const uint32_t slot = k % static_cast<uint32_t>(stages);
  const uint32_t round = k / static_cast<uint32_t>(stages);
  if (round > 0 && !mbar_wait(&empty[slot], (round - 1u) & 1u, kSiteEmpty)) return false;
  desc[slot].flags = kDone;
  mbar_arrive(&full[slot]);
  ++k;
  return true;
}

// ---------------------------------------------------------------------------
// Consumer side
// ---------------------------------------------------------------------------

// Folds the blocks of one stage that belong to this warp into keys[c0 + b].
//
// Lane per block (the common block sizes, see fold_stage): a warp takes 32
// consecutive blocks at a time and lane l folds block 32g + l on its own,
// over every piece, with no exchange between lanes. Lane l visits the
// elements of its block in its own order: element i ^ l for blocks of 32 or
// more (i ^ l stays inside the same aligned run of 32), (i + l / (32 / bs))
// mod bs for smaller ones. The 32 lanes of every load then ask for 32
// different banks whatever the pieces' alignment (checked exhaustively on the
// CPU for every block size and offset, fp32; bf16 lanes pair up on words).
// A lane keeps a whole block's loads in flight, and each key is stored once.
// Groups go to the consumer warps in turn across stages (`gbase`: groups in
// the earlier stages).
// MERGE: several stages hold pieces of the same blocks (one shard each), so
// keys are merged with atomicMax into keys that start at key(-inf).
template <typename E, int BS, bool MERGE>
__device__ __forceinline__ void fold_lane_blocks(const unsigned char* stage, const StageDesc& d,
                                                 int g0, int gstep,
                                                 uint32_t* __restrict__ keys) {
  constexpr int ES = E::kBytes;
  constexpr int T = BS < 32 ? BS : 32;  // offsets in the lane's table
  constexpr int CH = BS < 32 ? 1 : BS / 32;
  constexpr int LB = BS <= 1 ? 0 : BS == 2 ? 1 : BS == 4 ? 2 : BS == 8 ? 3 : 4;
  const int lane = threadIdx.x & 31;
  // The descriptor's fields in registers: key stores may alias shared
  // memory, so the compiler would reload them on every block.
  const int32_t c0 = d.c0, n = d.n, cnt = d.cnt;
  const unsigned char* __restrict__ const piece = stage + d.off;
  // Byte offsets of this lane's visiting order within a run of T elements.
  uint32_t offs[T];
#pragma unroll
  for (int i = 0; i < T; ++i)
    offs[i] = static_cast<uint32_t>(BS >= 32 ? (i ^ lane) : ((i + (lane >> (5 - LB))) & (BS - 1))) *
              ES;
  const int32_t ngroups = (n + 31) >> 5;
  for (int32_t g = g0; g < ngroups; g += gstep) {
    const int32_t blk = g * 32 + lane;
    if (blk >= n) continue;
    float acc[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
    {
      const int32_t valid = cnt - blk * BS;
      if (valid <= 0) continue;
      const unsigned char* pb = piece + static_cast<uint32_t>(blk * BS) * ES;
      if (valid >= BS) {
#pragma unroll
        for (int i = 0; i < T; ++i)
#pragma unroll
          for (int c = 0; c < CH; ++c)
            acc[(i + c) & 3] =
                max_nan(acc[(i + c) & 3], stage_elem<E>(pb + offs[i] + c * 32 * ES));
      } else {
        // The window's last block: only its first `valid` elements.
        for (int32_t e = 0; e < valid; ++e) acc[0] = max_nan(acc[0], stage_elem<E>(pb + e * ES));
      }
    }
    const uint32_t key = order_key(max_nan(max_nan(acc[0], acc[1], acc[2]), acc[3]));
    if (MERGE)
      atomicMax(&keys[c0 + blk], key);
    else
      keys[c0 + blk] = key;
  }
}

// The same with 16-byte loads, for a piece whose first element sits on a
// 16-byte boundary of the stage and blocks of whole 16-byte chunks (CH per
// block): lane l reads chunk c ^ (l & 7) of its block (8 chunks or more) or
// (c + l / (8 / CH)) mod CH (fewer), so that every 8-lane phase of a 16-byte
// load spreads over the 8 bank groups (checked exhaustively on the CPU). A
// chunk is four fp32 values, or eight bf16 values folded in pairs with
// max.NaN.bf16x2 and widened once per block.
template <typename E, int BS, bool MERGE>
__device__ __forceinline__ void fold_lane_blocks_vec(const unsigned char* stage,
                                                     const StageDesc& d, int g0, int gstep,
                                                     uint32_t* __restrict__ keys) {
  constexpr int ES = E::kBytes;
  constexpr int CH = BS * ES / 16;
  static_assert(CH >= 1 && (BS * ES) % 16 == 0, "whole 16-byte chunks");
  constexpr int SH = CH >= 8 ? 0 : CH == 4 ? 1 : CH == 2 ? 2 : 3;
  const int lane = threadIdx.x & 31;
  // The descriptor's fields in registers: key stores may alias shared
  // memory, so the compiler would reload them on every block.
  const int32_t c0 = d.c0, n = d.n, cnt = d.cnt;
  const unsigned char* __restrict__ const piece = stage + d.off;
  uint32_t offs[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c)
    offs[c] = static_cast<uint32_t>(CH >= 8 ? (c ^ (lane & 7)) : ((c + (lane >> SH)) % CH)) * 16;
  const int32_t ngroups = (n + 31) >> 5;
  for (int32_t g = g0; g < ngroups; g += gstep) {
    const int32_t blk = g * 32 + lane;
    if (blk >= n) continue;
    const int32_t valid = cnt - blk * BS;
    if (valid <= 0) continue;
    const unsigned char* pb = piece + static_cast<uint32_t>(blk * BS) * ES;
    float acc;
    if (valid >= BS) {
      if constexpr (ES == 4) {
        float a4[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(pb + offs[c]);
          a4[(c & 1) * 2] = max_nan(a4[(c & 1) * 2], v.x, v.y);
          a4[(c & 1) * 2 + 1] = max_nan(a4[(c & 1) * 2 + 1], v.z, v.w);
        }
        acc = max_nan(max_nan(a4[0], a4[1], a4[2]), a4[3]);
      } else {
        uint32_t w[2] = {BF16::kNegInfWord, BF16::kNegInfWord};
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(pb + offs[c]);
          w[0] = max_nan_bf16x2(w[0], v.x);
          w[1] = max_nan_bf16x2(w[1], v.y);
          w[0] = max_nan_bf16x2(w[0], v.z);
          w[1] = max_nan_bf16x2(w[1], v.w);
        }
        const uint32_t m = max_nan_bf16x2(w[0], w[1]);
        acc = max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
      }
    } else {
      // The window's last block: only its first `valid` elements.
      acc = neg_inf();
      for (int32_t e = 0; e < valid; ++e) acc = max_nan(acc, stage_elem<E>(pb + e * ES));
    }
    const uint32_t key = order_key(acc);
    if (MERGE)
      atomicMax(&keys[c0 + blk], key);
    else
      keys[c0 + blk] = key;
  }
}

// Other block sizes: lanes on consecutive elements, unconditional loads (an
// index past a piece's end reads the piece's first element, inside the CTA's
// shared memory, and a select drops it), one warp reduction per block (a
// redux, or xor shuffles over bs lanes for blocks below 32).
template <typename E, bool MERGE>
__device__ __forceinline__ void fold_elems(const unsigned char* stage, const StageDesc& d,
                                           int32_t bs, int32_t bs_log2, int t0, int tstep,
                                           uint32_t* __restrict__ keys) {
  constexpr int ES = E::kBytes;
  const int lane = threadIdx.x & 31;
  // The descriptor's fields in registers: key stores may alias shared
  // memory, so the compiler would reload them on every block.
  const int32_t c0 = d.c0, n = d.n, cnt = d.cnt;
  const unsigned char* __restrict__ const piece = stage + d.off;
  if (bs >= 32) {
    for (int32_t b = t0; b < n; b += tstep) {
      float acc = neg_inf();
      for (int32_t i = 0; i < bs; i += 32) {
        const int32_t j = b * bs + i + lane;
        const int32_t lim = cnt;
        const float v = stage_elem<E>(piece + (j < lim ? j : 0) * ES);
        acc = j < lim ? max_nan(acc, v) : acc;
      }
      const uint32_t key = __reduce_max_sync(0xffffffffu, order_key(acc));
      if (lane == 0) {
        if (MERGE)
          atomicMax(&keys[c0 + b], key);
        else
          keys[c0 + b] = key;
      }
    }
  } else {
    const int32_t ntile = (n * bs + 31) >> 5;
    for (int32_t tt = t0; tt < ntile; tt += tstep) {
      const int32_t j = tt * 32 + lane;
      const int32_t lim = cnt;
      const float v = stage_elem<E>(piece + (j < lim ? j : 0) * ES);
      const float acc = j < lim ? v : neg_inf();
      uint32_t key = order_key(acc);
      for (int o = 1; o < bs; o <<= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
      const int32_t blk = j >> bs_log2;
      if ((lane & (bs - 1)) == 0 && blk < n) {
        if (MERGE)
          atomicMax(&keys[c0 + blk], key);
        else
          keys[c0 + blk] = key;
      }
    }
  }
}

// Whether a block size takes the lane-per-block path (one piece per stage in
// every mode).
__host__ __device__ __forceinline__ bool lane_per_block(int32_t bs) {
  return bs >= 2 && bs <= 128 && (bs & (bs - 1)) == 0;
}

// Lane per block with 16-byte loads when the piece starts `off` bytes past a
// 16-byte boundary (0 < off < 16; every block then starts `off` bytes into
// a chunk, as a block is a whole number of chunks). A block covers its CH + 1
// chunks partly: its first chunk from byte off on, chunks 1 .. CH-1 whole,
// and its last chunk (the next block's first) below byte off. The two
// partial chunks are complementary, so one bit-select per word (bytes below
// off from the last chunk, the rest from the first) gives a full chunk of
// the block's own elements. The whole chunks are visited in a lane-rotated
// order, (c + lane % 8) mod (CH - 1), so that the 8 lanes of each 16-byte
// load phase mostly hit 8 different bank groups.
template <typename E, int BS, bool MERGE>
__device__ __forceinline__ void fold_lane_blocks_vmis(const unsigned char* stage,
                                                      const StageDesc& d, int g0, int gstep,
                                                      uint32_t* __restrict__ keys) {
  constexpr int ES = E::kBytes;
  constexpr int CH = BS * ES / 16;
  static_assert(CH >= 2 && (BS * ES) % 16 == 0, "at least two whole 16-byte chunks");
  const int lane = threadIdx.x & 31;
  const int32_t c0 = d.c0, n = d.n, cnt = d.cnt;
  const uint32_t off = d.off & 15u;
  const unsigned char* __restrict__ const base = stage + (d.off & ~15u);
  // Byte mask of the first chunk's part in word w: bytes at or past `off`.
  uint32_t m[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t mw = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) mw |= (4u * w + b >= off) ? (0xFFu << (8 * b)) : 0u;
    m[w] = mw;
  }
  const int rot = lane & 7;
  const int32_t ngroups = (n + 31) >> 5;
  for (int32_t g = g0; g < ngroups; g += gstep) {
    const int32_t blk = g * 32 + lane;
    if (blk >= n) continue;
    const int32_t valid = cnt - blk * BS;
    if (valid <= 0) continue;
    const unsigned char* pb = base + static_cast<uint32_t>(blk * BS) * ES;
    float acc;
    if (valid >= BS) {
      const uint4 f = *reinterpret_cast<const uint4*>(pb);
      const uint4 l = *reinterpret_cast<const uint4*>(pb + CH * 16);
      uint4 e;
      e.x = (f.x & m[0]) | (l.x & ~m[0]);
      e.y = (f.y & m[1]) | (l.y & ~m[1]);
      e.z = (f.z & m[2]) | (l.z & ~m[2]);
      e.w = (f.w & m[3]) | (l.w & ~m[3]);
      if constexpr (ES == 4) {
        float a4[4] = {max_nan(__uint_as_float(e.x), __uint_as_float(e.y)),
                       max_nan(__uint_as_float(e.z), __uint_as_float(e.w)), neg_inf(), neg_inf()};
#pragma unroll
        for (int c = 0; c < CH - 1; ++c) {
          int t = c + rot;
          t = t >= CH - 1 ? t - (CH - 1) : t;
          if (CH - 1 < 8) t = (c + rot) % (CH - 1);
          const float4 v = *reinterpret_cast<const float4*>(pb + 16 * (1 + t));
          a4[(c & 1) * 2] = max_nan(a4[(c & 1) * 2], v.x, v.y);
          a4[(c & 1) * 2 + 1] = max_nan(a4[(c & 1) * 2 + 1], v.z, v.w);
        }
        acc = max_nan(max_nan(a4[0], a4[1], a4[2]), a4[3]);
      } else {
        uint32_t w2[2] = {max_nan_bf16x2(e.x, e.z), max_nan_bf16x2(e.y, e.w)};
#pragma unroll
        for (int c = 0; c < CH - 1; ++c) {
          int t = c + rot;
          t = t >= CH - 1 ? t - (CH - 1) : t;
          if (CH - 1 < 8) t = (c + rot) % (CH - 1);
          const uint4 v = *reinterpret_cast<const uint4*>(pb + 16 * (1 + t));
          w2[0] = max_nan_bf16x2(w2[0], v.x);
          w2[1] = max_nan_bf16x2(w2[1], v.y);
          w2[0] = max_nan_bf16x2(w2[0], v.z);
          w2[1] = max_nan_bf16x2(w2[1], v.w);
        }
        const uint32_t mm = max_nan_bf16x2(w2[0], w2[1]);
        acc = max_nan(__uint_as_float(mm << 16), __uint_as_float(mm & 0xFFFF0000u));
      }
    } else {
      // The window's last block: only its first `valid` elements.
      acc = neg_inf();
      for (int32_t e = 0; e < valid; ++e) acc = max_nan(acc, stage_elem<E>(pb + off + e * ES));
    }
    const uint32_t key = order_key(acc);
    if (MERGE)
      atomicMax(&keys[c0 + blk], key);
    else
      keys[c0 + blk] = key;
  }
}

// The warp's share of one stage: the lane-per-block groups (gbase + g) %
// gstep == g0, or every gstep-th block / tile of the element path. VMIS:
// pieces off the 16-byte grid fold with 16-byte loads (fold_lane_blocks_vmis;
// the cooperative kernel, where folding warps share the stage) rather than
// element loads (the per-warp kernel, where the two partial chunks' bank
// conflicts sit on the warp's own path: prefill 35.0 -> 37.5 us with them).
template <typename E, int MODE, bool VMIS>
__device__ __forceinline__ void fold_stage(const PipeArgs& a, const unsigned char* stage,
                                           const StageDesc& d, int g0, int gstep, uint32_t gbase,
                                           uint32_t* __restrict__ keys) {
  constexpr bool M = MODE != kPipeUnsharded;  // one shard per stage: merge
  constexpr int ES = E::kBytes;
  const int first = static_cast<int>((static_cast<uint32_t>(g0) + gstep - gbase % gstep) % gstep);
  if ((d.off & 15u) == 0) {
    // The piece starts on a 16-byte boundary: whole 16-byte chunks per block.
    switch (a.block_size) {
      case 4:
        if constexpr (ES == 4) {
          fold_lane_blocks_vec<E, 4, M>(stage, d, first, gstep, keys);
          return;
        }
        break;
      case 8: fold_lane_blocks_vec<E, 8, M>(stage, d, first, gstep, keys); return;
      case 16: fold_lane_blocks_vec<E, 16, M>(stage, d, first, gstep, keys); return;
      case 32: fold_lane_blocks_vec<E, 32, M>(stage, d, first, gstep, keys); return;
      case 64: fold_lane_blocks_vec<E, 64, M>(stage, d, first, gstep, keys); return;
      case 128: fold_lane_blocks_vec<E, 128, M>(stage, d, first, gstep, keys); return;
      default: break;
    }
  }
  if (VMIS && a.block_size * ES >= 32) {
    // Off the 16-byte grid: 16-byte loads, the two partial chunks combined.
    switch (a.block_size) {
      case 8:
        if constexpr (ES == 4) {
          fold_lane_blocks_vmis<E, 8, M>(stage, d, first, gstep, keys);
          return;
        }
        break;
      case 16: fold_lane_blocks_vmis<E, 16, M>(stage, d, first, gstep, keys); return;
      case 32: fold_lane_blocks_vmis<E, 32, M>(stage, d, first, gstep, keys); return;
      case 64: fold_lane_blocks_vmis<E, 64, M>(stage, d, first, gstep, keys); return;
      case 128: fold_lane_blocks_vmis<E, 128, M>(stage, d, first, gstep, keys); return;
      default: break;
    }
  }
  switch (a.block_size) {
    case 2: fold_lane_blocks<E, 2, M>(stage, d, first, gstep, keys); return;
    case 4: fold_lane_blocks<E, 4, M>(stage, d, first, gstep, keys); return;
    case 8: fold_lane_blocks<E, 8, M>(stage, d, first, gstep, keys); return;
    case 16: fold_lane_blocks<E, 16, M>(stage, d, first, gstep, keys); return;
    case 32: fold_lane_blocks<E, 32, M>(stage, d, first, gstep, keys); return;
    case 64: fold_lane_blocks<E, 64, M>(stage, d, first, gstep, keys); return;
    case 128: fold_lane_blocks<E, 128, M>(stage, d, first, gstep, keys); return;
    default: fold_elems<E, M>(stage, d, a.block_size, a.bs_log2, g0, gstep, keys); return;
  }
}

// Lane-per-block groups in a stage of n blocks (0 for the element path,
// whose work is split by block or tile and needs no rotation).
__device__ __forceinline__ uint32_t stage_groups(int32_t bs, int32_t n) {
  return lane_per_block(bs) ? static_cast<uint32_t>((n + 31) >> 5) : 0u;
}

// The keys of a part [b0, b1) of a row that is split over several units:
// published to the workspace; the last part to arrive reads the others back
// and goes on to rank (returns true to every consumer thread).
template <typename Sync>
__device__ __forceinline__ bool merge_parts(const PipeArgs& a, int32_t row, int32_t nblk,
                                            int32_t b0, int32_t b1, int32_t parts, uint32_t* keys,
                                            int* s_last) {
  uint32_t* wrow = a.ws_keys + static_cast<int64_t>(row) * a.nb;
  for (int32_t b = b0 + Sync::tid(); b < b1; b += Sync::count()) __stcg(wrow + b, keys[b]);
  __threadfence();
  Sync::sync();
  if (Sync::tid() == 0) {
    // Count this part in; a counter word can hold an earlier call's block key
    // (>= key(-inf)), which reads as zero. Each failed CAS but the first
    // means another part arrived, so parts + 1 attempts suffice.
    uint32_t* counter = a.ws_count + row;
    uint32_t seen = 0u;
    int last = 0;
    for (int32_t i = 0; i < parts + 2; ++i) {
      const uint32_t count = (seen >= kKeyNegInf ? 0u : seen) + 1u;
      const uint32_t want = count == static_cast<uint32_t>(parts) ? 0u : count;
      const uint32_t prev = atomicCAS(counter, seen, want);
      if (prev == seen) {
        last = count == static_cast<uint32_t>(parts);
        break;
      }
      seen = prev;
    }
    *s_last = last;
  }
  Sync::sync();
  if (!*s_last) return false;
  __threadfence();
  for (int32_t b = Sync::tid(); b < nblk; b += Sync::count())
    if (b < b0 || b >= b1) keys[b] = __ldcg(wrow + b);
  return true;
}

template <typename E>
__device__ __forceinline__ typename E::T* score_row(const PipeArgs& a, int32_t row) {
  return a.scores ? static_cast<typename E::T*>(a.scores) + static_cast<int64_t>(row) * a.ld_scores
                  : nullptr;
}

// After a CTA's last (failing) take: the last CTA to finish resets the queue.
__device__ __forceinline__ void retire_queue(const PipeArgs& a) {
  if (!a.queue) return;
  __threadfence();
  if (atomicAdd(a.queue + 1, 1u) == gridDim.x - 1u) {
    atomicExch(a.queue, 0u);
    atomicExch(a.queue + 1, 0u);
  }
}

// Longest rows first (on request; index order is the default, see
// launch_coop_nw). With rows handed out by the unit counter, CTAs that start
// on long rows and pick up short ones when they free up finish close
// together (greedy list scheduling in longest-first order). Every CTA computes
// the same order: a stable counting sort of the rows by window length, cut
// into kLptClasses classes of width/(kLptClasses - 1) elements, longest class
// first and row index ascending within a class. Warp w sorts a contiguous
// range of 32-row chunks; __match_any_sync gives each lane its peers in the
// same class. Scratch (per-warp class counts, the class starts and the rows'
// classes) lives in the ring, which no copy touches before the order is
// built.
constexpr int kLptClasses = 128;
constexpr int kLptMaxRows = 4096;

__host__ __device__ __forceinline__ size_t lpt_scratch_bytes(int warps, int32_t rows) {
  return static_cast<size_t>(warps + 1) * kLptClasses * 4 + static_cast<size_t>(rows);
}

template <int NWARPS>
__device__ void longest_first_order(const PipeArgs& a, uint16_t* __restrict__ order,
                                    unsigned char* __restrict__ scratch) {
  uint32_t* hist = reinterpret_cast<uint32_t*>(scratch);  // [NWARPS][kLptClasses]
  uint32_t* start = hist + NWARPS * kLptClasses;           // [kLptClasses]
  unsigned char* cls = reinterpret_cast<unsigned char*>(start + kLptClasses);  // [rows]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < NWARPS * kLptClasses; i += blockDim.x) hist[i] = 0u;
  const int32_t rows = a.rows;
  // Every row's class (independent loads, all in flight together).
  const uint64_t width = static_cast<uint64_t>(max(a.width, 1));
#pragma unroll 4
  for (int32_t r = threadIdx.x; r < rows; r += blockDim.x) {
    const Bounds bnd = load_bounds<kPipeUnsharded>(a, r);
    const int32_t e = min(bnd.hi, a.width);
    const int32_t st = min(max(bnd.lo, 0), e);
    const uint64_t n = e > st ? static_cast<uint64_t>(e - st) : 0u;
    cls[r] = static_cast<unsigned char>((kLptClasses - 1) -
                                        static_cast<int>(n * (kLptClasses - 1) / width));
  }
  __syncthreads();
  const int32_t nch = (rows + 31) >> 5;
  const int32_t cpw = (nch + NWARPS - 1) / NWARPS;
  const int32_t c0 = warp * cpw, c1 = min(c0 + cpw, nch);
  uint32_t* h = hist + warp * kLptClasses;
  for (int32_t c = c0; c < c1; ++c) {
    const int32_t r = c * 32 + lane;
    const int b = r < rows ? static_cast<int>(cls[r]) : -1;  // 0: longest
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    if (b >= 0 && lane == __ffs(peers) - 1) h[b] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // Each class's start in the order (an exclusive scan over classes, longest
  // first), then each warp's start within the class: one thread per class
  // sums the warps' counts, warp 0 scans the sums, one thread per class
  // turns its counts into offsets (short independent chains, not one long
  // one).
  for (int b = threadIdx.x; b < kLptClasses; b += blockDim.x) {
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) t += hist[w * kLptClasses + b];
    start[b] = t;
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int PER = kLptClasses / 32;
    uint32_t t[PER], sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      t[i] = start[lane * PER + i];
      sum += t[i];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    uint32_t run = incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      start[lane * PER + i] = run;
      run += t[i];
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kLptClasses; b += blockDim.x) {
    uint32_t c[NWARPS];
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) c[w] = hist[w * kLptClasses + b];
    uint32_t off = start[b];
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
      hist[w * kLptClasses + b] = off;
      off += c[w];
    }
  }
  __syncthreads();
  for (int32_t c = c0; c < c1; ++c) {
    const int32_t r = c * 32 + lane;
    const int b = r < rows ? static_cast<int>(cls[r]) : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    if (b >= 0) order[h[b] + __popc(peers & ((1u << lane) - 1u))] = static_cast<uint16_t>(r);
    __syncwarp();
    if (b >= 0 && lane == __ffs(peers) - 1) h[b] += __popc(peers);
    __syncwarp();
  }
  // The ring's generic-proxy accesses come before the copies that later
  // write it.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
}

// A finished unit handed from the fold warps to the rank warps.
struct UnitMeta {
  int32_t row, nblk, pin, b0, b1, parts, done;
};

constexpr int kRankWarps = 4;

// Shared memory of a coop CTA: ring, its barriers and descriptors, then two
// key buffers [nb] (padded to 4), the candidates [max(kpad, kRankMax)] and,
// with a.lpt, the row order [rows] (uint16).
__host__ __device__ __forceinline__ size_t coop_keys_offset(int stages, int stage_bytes) {
  return static_cast<size_t>(stages) * stage_bytes +
         ((static_cast<size_t>(stages) * (16 + sizeof(StageDesc)) + 127) & ~static_cast<size_t>(127));
}

// Warps 0 .. NW-1 fold, NW .. NW+3 rank, warp NW+4 produces. The fold warps
// fill one of two key buffers with a unit's block keys and hand it to the
// rank warps (mbarrier kfull, with the unit in `meta`); the rank warps merge
// split rows, pin, rank and store it, reset the buffer (key(-inf), in the
// shard forms whose stages merge into it) and hand it back (kempty), while
// the fold warps go on with the next unit in the other buffer. A row's top-k
// thus never stops the fold, and no barrier joins the fold warps.
template <typename E, int MODE, int NW>
__global__ void __launch_bounds__((NW + kRankWarps + 1) * 32, NW == 4 ? 2 : 1)
    pipe_coop_kernel(const PipeArgs a) {
  constexpr int NR = kRankWarps;
  using RankSync = NamedSync<NR * 32, 2, NW * 32>;
  constexpr bool kMerge = MODE != kPipeUnsharded;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(a.stages) * a.stage_bytes);
  uint64_t* empty = full + a.stages;
  StageDesc* desc = reinterpret_cast<StageDesc*>(empty + a.stages);
  const int32_t nbp = (a.nb + 3) & ~3;
  uint32_t* keys0 = reinterpret_cast<uint32_t*>(smem + coop_keys_offset(a.stages, a.stage_bytes));
  uint64_t* cand = reinterpret_cast<uint64_t*>(keys0 + 2 * nbp);
  uint16_t* order = reinterpret_cast<uint16_t*>(cand + max(a.kpad, kRankMax));
  __shared__ TopkShared tsh;
  __shared__ int s_last;
  __shared__ __align__(8) uint64_t kfull[2], kempty[2];
  __shared__ UnitMeta meta[2];
  __shared__ PieceTable pt;  // the producer's current unit

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int32_t b = threadIdx.x; b < 2 * nbp; b += blockDim.x) keys0[b] = kKeyNegInf;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], NW);
      mbar_init(&kempty[i], 1);
    }
    mbar_init_fence();
  }
  __syncthreads();
  // Whole unsharded rows from the unit counter: the producer claims a CTA's
  // next row only when the current row's last stage is due (the ring still
  // holds that row's last stages, which hides the claim's round trip), so
  // rows go to CTAs as they free up; CTA b starts with row b, so that its
  // first bound load waits on no claim. Claiming two ahead from the start
  // fixed each CTA's rows when the launch began (on decode one CTA drew two
  // of the longest rows, 480 KB against 194 KB on average): timed in turn,
  // decode 25.4 -> 23.4 us, long 65.6 -> 63.3 us, decode_bf16 20.6 -> 20.4 us.
  const bool claim_late = MODE == kPipeUnsharded && a.split == 1 && a.queue != nullptr &&
                          !a.claim_ahead;
  if constexpr (MODE == kPipeUnsharded)
    if (a.lpt) longest_first_order<NW + NR + 1>(a, order, ring);

  if (claim_late && warp == NW + NR) {
    const uint32_t total = static_cast<uint32_t>(a.rows);
    uint32_t u = blockIdx.x;  // the grid never exceeds the rows
    uint32_t k = 0;
    int ok = 1;
    while (ok && u < total) {
      const int32_t row = a.lpt ? static_cast<int32_t>(order[u]) : static_cast<int32_t>(u);
      const LanePlan<E> p = plan_lane<E, MODE>(a, row, load_bounds<MODE>(a, row), lane);
      if (lane == 0) {
        pt.origin[0] = reinterpret_cast<const unsigned char*>(p.origin);
        pt.len[0] = p.len;
        ok = emit_unit<E>(a, pt, 1, row, p.nblk, p.pin, 0, p.nblk, 1, ring, full, empty, desc,
                          a.stages, k, &u);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
    }
    if (lane == 0) {
      retire_queue(a);
      if (ok) emit_done(full, empty, desc, a.stages, k);
    }
    return;
  }

  if (warp == NW + NR) {
    // Producer warp for parts of rows, the shard forms and the fixed order.
    // Units are fetched two ahead: while the stages of unit u
    // go out, the bounds of the next unit and the index of the one after it
    // are in flight, so a unit boundary waits on no memory round trip.
    const uint32_t S = static_cast<uint32_t>(a.split);
    const uint32_t total = static_cast<uint32_t>(a.rows) * S;
    const int npieces = MODE == kPipeUnsharded ? 1 : a.shards;
    uint32_t u = 0, u1 = 0;
    if (lane == 0) {
      u = a.queue ? atomicAdd(a.queue, 1u) : blockIdx.x;
      u1 = a.queue ? atomicAdd(a.queue, 1u) : blockIdx.x + gridDim.x;
    }
    u = __shfl_sync(0xffffffffu, u, 0);
    u1 = __shfl_sync(0xffffffffu, u1, 0);
    Bounds bnd{0, 0};
    if (u < total) bnd = load_bounds<MODE>(a, static_cast<int32_t>(u / S));
    uint32_t k = 0;  // stages issued (lane 0)
    int ok = 1;
    while (ok && u < total) {
      Bounds nbnd{0, 0};
      if (u1 < total) nbnd = load_bounds<MODE>(a, static_cast<int32_t>(u1 / S));
      uint32_t u2 = 0;
      if (lane == 0) u2 = a.queue ? (u1 < total ? atomicAdd(a.queue, 1u) : u1) : u1 + gridDim.x;
      const int32_t row = static_cast<int32_t>(u / S);
      const int32_t part = static_cast<int32_t>(u % S);
      const LanePlan<E> p = plan_lane<E, MODE>(a, row, bnd, lane);
      int32_t b0 = 0, b1 = p.nblk, parts = 1;
      if (a.split > 1) {
        const int32_t per = max(kPartUnit, ((p.nblk + a.split - 1) / a.split + kPartUnit - 1) /
                                               kPartUnit * kPartUnit);
        parts = max(1, (p.nblk + per - 1) / per);
        b0 = min(part * per, p.nblk);
        b1 = min(b0 + per, p.nblk);
      }
      if (part < parts) {
        if (lane < npieces) {
          pt.origin[lane] = reinterpret_cast<const unsigned char*>(p.origin);
          pt.len[lane] = p.len;
        }
        __syncwarp();
        if (lane == 0)
          ok = emit_unit<E>(a, pt, npieces, row, p.nblk, p.pin, b0, b1, parts, ring, full, empty,
                            desc, a.stages, k);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();  // the table is read before it is rewritten
      }
      u = u1;
      bnd = nbnd;
      u1 = __shfl_sync(0xffffffffu, u2, 0);
    }
    if (lane == 0) {
      retire_queue(a);
      if (ok) emit_done(full, empty, desc, a.stages, k);
    }
    return;
  }

  if (warp >= NW) {
    // Rank warps: units in the order the fold warps finish them.
    uint32_t rounds0 = 0, rounds1 = 0;  // units taken from each buffer
    for (int rb = 0;; rb ^= 1) {
      uint32_t& rounds = rb ? rounds1 : rounds0;
      const bool ok = mbar_wait(&kfull[rb], rounds & 1u, kSiteKeys);
      if (!__all_sync(0xffffffffu, ok)) return;
      const UnitMeta m = meta[rb];
      if (m.done) return;
      uint32_t* keys = keys0 + rb * nbp;
      if (m.parts == 1 || merge_parts<RankSync>(a, m.row, m.nblk, m.b0, m.b1, m.parts, keys,
                                                &s_last)) {
        for (int32_t b = m.nblk + RankSync::tid(); b <= m.pin; b += RankSync::count())
          keys[b] = kKeyNegInf;
        RankSync::sync();
        const int32_t n_live = max(m.nblk, m.pin + 1), kk = min(a.topk, a.nb);
        int32_t* out = a.topk > 0 ? a.out + static_cast<int64_t>(m.row) * a.ld_out : nullptr;
        if (a.rank_warp && kk <= 32 && n_live <= 1024) {
          // One rank warp: fewer instructions, but a longer path than four
          // warps sharing the keys (decode 29.8 against 28.3 us).
          if (RankSync::tid() < 32)
            topk_warp_wide(keys, a.nb, n_live, kk, m.pin, cand, max(a.kpad, kRankMax), out,
                           a.topk, score_row<E>(a, m.row));
        } else {
          topk_store<typename E::T, RankSync>(keys, a.nb, n_live, kk, m.pin, cand, a.kpad, out,
                                              a.topk, score_row<E>(a, m.row), tsh);
        }
      }
      RankSync::sync();  // every rank thread is done with the keys
      if (kMerge) {
        for (int32_t b = RankSync::tid(); b < a.nb; b += RankSync::count()) keys[b] = kKeyNegInf;
        RankSync::sync();
      }
      if (RankSync::tid() == 0) mbar_arrive(&kempty[rb]);
      ++rounds;
    }
  }

  // Fold warps.
  uint32_t gbase = 0;        // lane-per-block groups in the stages before this one
  int ub = 0;                // key buffer of the current unit
  uint32_t uses0 = 0, uses1 = 0;
  bool have = false;         // the current unit's buffer is ours
  for (uint32_t k = 0;; ++k) {
    const uint32_t slot = k % static_cast<uint32_t>(a.stages);
    // A phase that never completes (a fault in the byte accounting) makes
    // every waiter give up; the warp leaves as one.
    const bool ok = mbar_wait(&full[slot], (k / static_cast<uint32_t>(a.stages)) & 1u, kSiteFull);
    if (!__all_sync(0xffffffffu, ok)) return;
    if (!have) {
      const uint32_t uses = ub ? uses1 : uses0;
      const bool free_ok = uses == 0 || mbar_wait(&kempty[ub], (uses - 1u) & 1u, kSiteKeys);
      if (!__all_sync(0xffffffffu, free_ok)) return;
      have = true;
    }
    const StageDesc& d = desc[slot];
    const int32_t flags = d.flags;
    if (flags & kDone) {
      // The done marker goes to the rank warps through the next buffer.
      if (warp == 0 && lane == 0) meta[ub].done = 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&kfull[ub]);
      return;
    }
    const int32_t row = d.row, nblk = d.nblk, pin = d.pin, b0 = d.b0, b1 = d.b1,
                  parts = d.parts;
    uint32_t* keys = keys0 + ub * nbp;
    if (!a.own_stages)
      fold_stage<E, MODE, true>(a, ring + static_cast<size_t>(slot) * a.stage_bytes, d, warp, NW,
                                gbase, keys);
    else if (k % NW == static_cast<uint32_t>(warp))
      fold_stage<E, MODE, true>(a, ring + static_cast<size_t>(slot) * a.stage_bytes, d, 0, 1, 0u,
                                keys);
    gbase += stage_groups(a.block_size, d.n);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (!(flags & kLast)) continue;
    if (warp == 0 && lane == 0) meta[ub] = UnitMeta{row, nblk, pin, b0, b1, parts, 0};
    __syncwarp();  // this warp's keys (and the unit) before the hand-over
    if (lane == 0) mbar_arrive(&kfull[ub]);
    if (ub) ++uses1; else ++uses0;
    ub ^= 1;
    have = false;
  }
}

// Shared memory of a solo CTA: NW rings of `stages`, their full barriers and
// descriptors, then per warp its keys [nb] and candidates [kWarpCand].
__host__ __device__ __forceinline__ size_t solo_warp_offset(int nw, int stages, int stage_bytes) {
  const size_t nst = static_cast<size_t>(nw) * stages;
  return nst * stage_bytes + ((nst * (8 + sizeof(StageDesc)) + 127) & ~static_cast<size_t>(127));
}
__host__ __device__ __forceinline__ size_t solo_warp_bytes(int32_t nb) {
  return static_cast<size_t>(kWarpCand) * 8 + static_cast<size_t>((nb + 3) & ~3) * 4;
}

// One stage of an unsharded row for a warp that produces for itself: lane
// 0 copies blocks [c, c + n) of the window and arms the stage's barrier.
template <typename E>
__device__ __forceinline__ void solo_emit(const PipeArgs& a, const LanePlan<E>& p, int32_t row,
                                          int32_t c, int32_t n, bool last,
                                          unsigned char* buf, uint64_t* full, StageDesc& d) {
  const int32_t j0 = c * a.block_size;
  const int32_t j1 = min((c + n) * a.block_size, p.len);
  uintptr_t A = 0;
  uint32_t bytes = 0, head = 0;
  if (j1 > j0) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p.origin + j0);
    const uintptr_t hi = reinterpret_cast<uintptr_t>(p.origin + j1);
    A = lo & ~static_cast<uintptr_t>(15);
    bytes = static_cast<uint32_t>(((hi + 15) & ~static_cast<uintptr_t>(15)) - A);
    head = static_cast<uint32_t>(lo - A);
  }
  d.row = row;
  d.c0 = c;
  d.n = n;
  d.flags = last ? kLast : 0;
  d.npieces = 1;
  d.nblk = p.nblk;
  d.pin = p.pin;
  d.b0 = 0;
  d.b1 = p.nblk;
  d.parts = 1;
  d.off = head;
  d.cnt = j1 > j0 ? j1 - j0 : 0;
  if (bytes > 0) {
    mbar_arrive_expect_tx(full, bytes);
    bulk_load(buf, reinterpret_cast<const void*>(A), bytes, full);
  } else {
    mbar_arrive(full);
  }
}

// One row per warp, each warp its own producer: warp g of the grid takes rows
// g, g + G, ... (G warps in all). Lane 0 keeps the warp's ring full: it
// issues the stages of the rows ahead (fetching each next row's bounds while
// the current one goes out) whenever a slot is free, so the copies of the
// next rows are in flight while the warp folds and ranks this one. A slot is
// free once the warp has folded it (the warp's own program order, with a
// __syncwarp before lane 0 reuses it), so no empty barriers are needed and no
// warp waits for another.
template <typename E, int NW>
__global__ void __launch_bounds__(NW * 32, 2) pipe_solo_kernel(const PipeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int nst = NW * a.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* ring = smem + static_cast<size_t>(warp) * a.stages * a.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nst) * a.stage_bytes) +
                   warp * a.stages;
  StageDesc* desc = reinterpret_cast<StageDesc*>(
                        reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nst) * a.stage_bytes) +
                        nst) +
                    warp * a.stages;
  unsigned char* wbase = smem + solo_warp_offset(NW, a.stages, a.stage_bytes);
  uint64_t* cand = reinterpret_cast<uint64_t*>(wbase + static_cast<size_t>(warp) * solo_warp_bytes(a.nb));
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + kWarpCand);
  if (lane == 0) {
    for (int i = 0; i < a.stages; ++i) mbar_init(&full[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  const uint32_t rows = static_cast<uint32_t>(a.rows);
  const uint32_t G = gridDim.x * NW;
  // Producer state (lane 0's values are the ones used): the row being issued,
  // its plan, the next block to issue, and the next row's bounds.
  uint32_t prow = blockIdx.x * NW + warp;
  Bounds bnd{0, 0}, nbnd{0, 0};
  if (prow < rows) bnd = load_bounds<kPipeUnsharded>(a, static_cast<int32_t>(prow));
  if (prow + G < rows) nbnd = load_bounds<kPipeUnsharded>(a, static_cast<int32_t>(prow + G));
  LanePlan<E> p = plan_lane<E, kPipeUnsharded>(a, static_cast<int32_t>(prow), bnd, 0);
  int32_t pc = 0;
  uint32_t kp = 0;  // stages issued
  for (uint32_t kc = 0;; ++kc) {
    // Issue while slots are free and rows remain.
    if (lane == 0) {
      while (prow < rows && kp - kc < static_cast<uint32_t>(a.stages)) {
        const uint32_t slot = kp % static_cast<uint32_t>(a.stages);
        const int32_t n = min(a.cap, p.nblk - pc);
        const bool last = pc + n >= p.nblk;
        solo_emit<E>(a, p, static_cast<int32_t>(prow), pc, n, last,
                     ring + static_cast<size_t>(slot) * a.stage_bytes, &full[slot], desc[slot]);
        ++kp;
        pc += n;
        if (last) {
          prow += G;
          pc = 0;
          if (prow < rows) {
            p = plan_lane<E, kPipeUnsharded>(a, static_cast<int32_t>(prow), nbnd, 0);
            if (prow + G < rows) nbnd = load_bounds<kPipeUnsharded>(a, static_cast<int32_t>(prow + G));
          }
        }
      }
    }
    kp = __shfl_sync(0xffffffffu, kp, 0);
    if (kc >= kp) break;  // nothing issued beyond what was consumed: done
    const uint32_t slot = kc % static_cast<uint32_t>(a.stages);
    const bool ok = mbar_wait(&full[slot], (kc / static_cast<uint32_t>(a.stages)) & 1u, kSiteFull);
    if (!__all_sync(0xffffffffu, ok)) return;
    const StageDesc& d = desc[slot];
    const int32_t flags = d.flags;
    const int32_t row = d.row, nblk = d.nblk, pin = d.pin;
    fold_stage<E, kPipeUnsharded, false>(a, ring + static_cast<size_t>(slot) * a.stage_bytes, d,
                                         0, 1, 0u, keys);
    __syncwarp();  // the slot and its descriptor are free for lane 0
    if (!(flags & kLast)) continue;
    // The lane-maximum bound: on the warp's own path it measured as fast as
    // topk_warp_wide's tighter bound (prefill 34.9 against 35.4 us), whose
    // rounds of warp maxima sit on that path.
    topk_warp(keys, a.nb, nblk, min(a.topk, a.nb), pin, cand,
              a.topk > 0 ? a.out + static_cast<int64_t>(row) * a.ld_out : nullptr, a.topk,
              score_row<E>(a, row));
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

std::atomic<int> g_over[16];

int sm_count_now() {
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

int max_smem_optin() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      n = 0;
    cached[dev] = n;
  }
  return cached[dev];
}

int max_smem_per_sm() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess)
      n = 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Remembers the largest dynamic shared memory set per (kernel, device).
std::mutex g_attr_mu;
struct AttrEntry {
  const void* fn;
  int dev;
  size_t bytes;
};
AttrEntry g_attr[64];
int g_attr_n = 0;

template <typename K>
cudaError_t opt_in_smem(K kernel, size_t bytes) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const void* fn = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (int i = 0; i < g_attr_n; ++i)
    if (g_attr[i].fn == fn && g_attr[i].dev == dev) {
      if (g_attr[i].bytes >= bytes) return cudaSuccess;
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(bytes));
      if (err == cudaSuccess) g_attr[i].bytes = bytes;
      return err;
    }
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
  if (err == cudaSuccess && g_attr_n < 64) g_attr[g_attr_n++] = {fn, dev, bytes};
  return err;
}

constexpr int kSoloWarps = 8;

bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int64_t x) {
  int l = 0;
  while ((int64_t(1) << (l + 1)) <= x) ++l;
  return l;
}

bool logits_on_device(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice;
}

// Whether to hand short unsharded rows one per warp.
bool want_solo(const PipeCall& c) {
  const int forced = g_over[DSA_LAUNCH_PIPELINE].load(std::memory_order_relaxed);
  if (forced == 2) return false;
  const bool fits = c.mode == kPipeUnsharded && c.topk <= 32 && c.nb <= 2048;
  if (forced == 3) return fits;
  return fits && static_cast<int64_t>(c.width) * c.elem_bytes <= 64 * 1024 &&
         c.rows >= 8 * static_cast<int64_t>(sm_count_now());
}

}  // namespace

void pipe_set_override(int knob, int value) {
  if (knob >= 0 && knob < 16) g_over[knob].store(value);
}
int pipe_get_override(int knob) { return (knob >= 0 && knob < 16) ? g_over[knob].load() : 0; }

bool pipe_takes(const PipeCall& c) {
  const int forced = g_over[DSA_LAUNCH_PIPELINE].load(std::memory_order_relaxed);
  if (forced == 1) return false;
  // The shard forms stay on select_kernel unless the pipelined kernels are
  // asked for: there select_kernel's eight shard streams per CTA measured
  // faster (DCP 85.8 us against 116 us and more).
  if (c.mode != kPipeUnsharded && forced == 0) return false;
  const int32_t bs = c.block_size;
  if (!(bs % 32 == 0 || (pow2(bs) && bs < 32))) return false;
  if (c.shards > kMaxShardLanes || c.nb > kPipeMaxBlocks || c.topk > kPipeMaxTopk) return false;
  if (c.rows * 8 > INT32_MAX) return false;
  if (static_cast<int64_t>(bs) * c.elem_bytes > 4096) return false;
  return logits_on_device(c.logits);
}

namespace {

// Shared memory a CTA may use when `ctas` of them share an SM (each CTA
// also pays the SM's 1 KiB reservation), less `static_bytes` of static
// shared memory.
size_t smem_budget(int ctas, size_t static_bytes) {
  const size_t per_sm = static_cast<size_t>(max_smem_per_sm());
  const size_t per_cta = std::min<size_t>(static_cast<size_t>(max_smem_optin()),
                                          per_sm / ctas - 1024);
  return per_cta > static_bytes + 64 ? per_cta - static_bytes - 64 : 0;
}

template <typename E, int MODE, int NW>
dsa_status launch_coop_nw(PipeArgs a, int64_t max_row_bytes, bool have_ws, int ctas,
                          cudaStream_t s) {
  const int sms = sm_count_now();
  const int pieces = 1;  // one piece per stage (one shard in the shard forms)
  const int slots = sms * ctas;
  // Parts per row: only when there are fewer rows than CTAs, never below
  // 64 KiB per part, at most 8; only with a workspace. (Merging parts costs
  // each part a fence, an atomic and a read-back: decode measured 30.7 us
  // unsplit against 45 us in 4 parts.)
  int split = 1;
  if (have_ws) {
    while (split < 8 && a.rows * split < slots && max_row_bytes / (2 * split) >= 64 * 1024)
      split <<= 1;
    const int forced = g_over[DSA_LAUNCH_PIPE_SPLIT].load(std::memory_order_relaxed);
    if (forced >= 1 && forced <= 8) split = forced;
  }
  a.split = split;
  a.own_stages = g_over[DSA_LAUNCH_PIPE_STAGE_OWNER].load(std::memory_order_relaxed) == 1;
  a.rank_warp = g_over[DSA_LAUNCH_RANK_CTA].load(std::memory_order_relaxed) == 2;
  // Longest rows first only on request (unsharded, unsplit, through the unit
  // counter): timed in turn on the same buffers, the ordering pass (about 2.5
  // us at the start of a flushed step) costs more than the balance gains:
  // decode 25.6 us in index order against 27.6 us longest first,
  // decode_bf16 20.6 against 23.1 us, long 65.6 us either way.
  const int ord = g_over[DSA_LAUNCH_PIPE_ORDER].load(std::memory_order_relaxed);
  a.lpt = MODE == kPipeUnsharded && split == 1 && a.queue != nullptr && a.rows <= kLptMaxRows &&
          ord == 2;
  a.claim_ahead = ord == 3;
  const size_t tail = 2 * static_cast<size_t>((a.nb + 3) & ~3) * 4 +
                      static_cast<size_t>(std::max(a.kpad, kRankMax)) * 8 +
                      (a.lpt ? ((static_cast<size_t>(a.rows) * 2 + 15) & ~static_cast<size_t>(15)) : 0);
  const size_t limit =
      smem_budget(ctas, sizeof(TopkShared) + sizeof(PieceTable) + 2 * sizeof(UnitMeta) + 128);
  // A stage carries `payload` bytes of whole blocks; its buffer adds 32 bytes
  // for the 16-byte rounding at both ends of the piece. The largest payload
  // of 48 (64 at one CTA per SM), 32 and 16 KiB that leaves room for two
  // stages: fewer, larger stages measured faster (48 against 32 KiB: decode
  // 28.0 -> 26.8 us, decode_bf16 21.2 -> 20.5 us, long 70.0 -> 69.3 us).
  const int kb = g_over[DSA_LAUNCH_PIPE_STAGE_KB].load(std::memory_order_relaxed);
  int stages = 0;
  for (int p = ctas == 1 ? 64 : 48; p >= 16 && stages < 2; p -= 16) {
    const int payload = (kb >= 4 && kb <= 64 ? kb : p) * 1024;
    a.stage_bytes = (payload + 32 * pieces + 127) & ~127;
    a.cap = static_cast<int32_t>(payload /
                                 (static_cast<int64_t>(pieces) * a.block_size * E::kBytes));
    stages = 16;
    while (stages >= 2 && coop_keys_offset(stages, a.stage_bytes) + tail > limit) --stages;
    if (a.cap < 1) stages = 0;
    if (kb >= 4 && kb <= 64) break;
  }
  const int fst = g_over[DSA_LAUNCH_PIPE_STAGES].load(std::memory_order_relaxed);
  if (fst >= 2 && fst < stages) stages = fst;
  if (stages < 2) return kPipeDeclined;
  a.stages = stages;
  // The order pass's scratch lives in the ring.
  if (static_cast<size_t>(stages) * a.stage_bytes < lpt_scratch_bytes(NW + kRankWarps + 1, a.rows))
    a.lpt = 0;
  const size_t smem = coop_keys_offset(stages, a.stage_bytes) + tail;
  auto kernel = pipe_coop_kernel<E, MODE, NW>;
  if (opt_in_smem(kernel, smem) != cudaSuccess) return DSA_ECUDA;
  const int64_t units = a.rows * static_cast<int64_t>(split);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(units, slots));
  kernel<<<grid, (NW + kRankWarps + 1) * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

// Rows of more than 256 KiB run at one CTA per SM with 8 folding warps and
// three 64 KiB stages (192 KiB in flight per SM, one producer): long (1024
// rows of 256-512 KiB) 69.0 -> 65.6 us. Shorter rows keep two CTAs per SM
// with 4 folding warps each: decode (rows of up to 256 KiB) measured 28.2
// against 30.0 us in the one-CTA shape, decode_bf16 20.5 against 25.1 us.
template <typename E, int MODE>
dsa_status launch_coop(const PipeArgs& a, int64_t max_row_bytes, bool have_ws, cudaStream_t s) {
  const int warps = g_over[DSA_LAUNCH_PIPE_WARPS].load(std::memory_order_relaxed);
  const int fc = g_over[DSA_LAUNCH_PIPE_CTAS].load(std::memory_order_relaxed);
  if (warps == 8 || (warps == 0 && max_row_bytes > 256 * 1024))
    return launch_coop_nw<E, MODE, 8>(a, max_row_bytes, have_ws, 1, s);
  return launch_coop_nw<E, MODE, 4>(a, max_row_bytes, have_ws, fc >= 1 ? std::min(fc, 2) : 2, s);
}

// Solo launch with `ctas` CTAs per SM; kPipeDeclined (nothing enqueued) when
// the rings and the warps' keys do not fit.
template <typename E>
dsa_status launch_solo_ctas(PipeArgs a, int ctas, cudaStream_t s) {
  const int sms = sm_count_now();
  const int kb = g_over[DSA_LAUNCH_PIPE_STAGE_KB].load(std::memory_order_relaxed);
  const size_t limit = smem_budget(ctas, 0);
  const size_t fixed = static_cast<size_t>(kSoloWarps) * solo_warp_bytes(a.nb);
  a.split = 1;
  a.queue = nullptr;
  // Stages of 8 KiB (4 KiB when two per warp do not fit), up to 4 per warp.
  int stages = 0;
  for (int payload = kb >= 4 && kb <= 64 ? kb * 1024 : 8192; payload >= 4096; payload /= 2) {
    a.stage_bytes = (payload + 32 + 127) & ~127;
    a.cap = static_cast<int32_t>(payload / (static_cast<int64_t>(a.block_size) * E::kBytes));
    stages = 4;
    while (stages >= 2 && solo_warp_offset(kSoloWarps, stages, a.stage_bytes) + fixed > limit)
      --stages;
    if ((stages >= 2 && a.cap >= 1) || kb != 0) break;
  }
  const int fst = g_over[DSA_LAUNCH_PIPE_STAGES].load(std::memory_order_relaxed);
  if (fst >= 2 && fst < stages) stages = fst;
  if (stages < 2 || a.cap < 1) return kPipeDeclined;
  a.stages = stages;
  const size_t smem = solo_warp_offset(kSoloWarps, stages, a.stage_bytes) + fixed;
  auto kernel = pipe_solo_kernel<E, kSoloWarps>;
  if (opt_in_smem(kernel, smem) != cudaSuccess) return DSA_ECUDA;
  const unsigned grid = static_cast<unsigned>(
      std::min<int64_t>((a.rows + kSoloWarps - 1) / kSoloWarps, static_cast<int64_t>(sms) * ctas));
  kernel<<<grid, kSoloWarps * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

// Two CTAs per SM (measured faster on packed prefill rows), one when the
// keys of rows with many blocks leave no room for two.
template <typename E>
dsa_status launch_solo(const PipeArgs& a, cudaStream_t s) {
  const int fc = g_over[DSA_LAUNCH_PIPE_CTAS].load(std::memory_order_relaxed);
  if (fc >= 1) return launch_solo_ctas<E>(a, std::min(fc, 2), s);
  const dsa_status st = launch_solo_ctas<E>(a, 2, s);
  return st == kPipeDeclined ? launch_solo_ctas<E>(a, 1, s) : st;
}

template <typename E>
dsa_status dispatch(const PipeCall& c, cudaStream_t s) {
  PipeArgs a{};
  a.logits = c.logits;
  a.ld = c.ld;
  a.shard_stride = c.shard_stride;
  a.shards = c.shards;
  a.width = c.width;
  a.row_ks = c.row_ks;
  a.row_ke = c.row_ke;
  a.row_repeat = c.row_repeat;
  a.block_size = c.block_size;
  a.bs_log2 = c.block_size < 32 ? log2i(c.block_size) : 0;
  a.global_block_size = c.global_block_size;
  a.nb = c.nb;
  a.nb_data = c.nb_data;
  a.pin_newest = c.pin_newest;
  a.topk = c.topk;
  int32_t kp = 1;
  while (kp < std::max<int32_t>(1, std::min(c.topk, c.nb))) kp <<= 1;
  a.kpad = kp;
  a.out = c.out;
  a.ld_out = c.ld_out;
  a.scores = c.scores;
  a.ld_scores = c.ld_scores;
  a.rows = static_cast<int32_t>(c.rows);
  // A workspace of full size gives split rows their keys and counters and,
  // unless a fixed order is forced, the unit queue.
  const bool have_ws = c.workspace && c.workspace_size >= ws_total_bytes(c.rows, c.nb);
  if (have_ws) {
    if (g_over[DSA_LAUNCH_PIPE_SCHED].load(std::memory_order_relaxed) != 1)
      a.queue = static_cast<uint32_t*>(c.workspace);
    a.ws_count = reinterpret_cast<uint32_t*>(static_cast<char*>(c.workspace) + ws_counts_offset());
    a.ws_keys = reinterpret_cast<uint32_t*>(static_cast<char*>(c.workspace) + ws_keys_offset(c.rows));
  }
  const int64_t max_row_bytes = static_cast<int64_t>(c.width) * c.elem_bytes * c.shards;
  if (want_solo(c)) {
    const dsa_status st = launch_solo<E>(a, s);
    if (st != kPipeDeclined) return st;
  }
  switch (c.mode) {
    case kPipeUnsharded: return launch_coop<E, kPipeUnsharded>(a, max_row_bytes, have_ws, s);
    case kPipeSharded: return launch_coop<E, kPipeSharded>(a, max_row_bytes, have_ws, s);
    default: return launch_coop<E, kPipeShardedStarts>(a, max_row_bytes, have_ws, s);
  }
}

}  // namespace

dsa_status pipe_select(const PipeCall& c, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return c.elem_bytes == 4 ? dispatch<F32>(c, s) : dispatch<BF16>(c, s);
}

}  // namespace dsa

extern "C" int dsa_pipeline_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, dsa::g_pipe_error, sizeof(v)) != cudaSuccess) return -1;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(dsa::g_pipe_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
  }
  return static_cast<int>(v);
}
