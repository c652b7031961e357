// mask.cu -- masking packed logits to the selected candidate blocks: the C
// ABI dsa_mask_candidate_logits[_sharded][_bf16] of include/dsa_cb.h.
//
// candidate_blocks.py diff, the masking function after selection: its
// docstring masks every packed logit outside the row's causal window or
// outside the row's request-local candidate blocks; under DCP the local
// block size is passed and the candidate ids apply unchanged.
// In place: logit c of a row becomes -inf when c is outside the row's window
// [s, e) or its request-local block (c - s) / block_size is not one of the
// row's candidate ids (ids < 0 are empty slots). Kept logits are not touched,
// so the pass never reads the logits: it only writes -inf. It is bound by
// HBM write bandwidth.
//
// One CTA per (shard, row, chunk of 32 KiB of logits). The chunk is cut
// into 16-byte-aligned slots (four fp32 or eight bf16 columns). Before any
// store, the CTA turns the row's candidate ids into two slot bitmaps in
// shared memory: `touch` (the slot holds at least one kept column) and
// `whole` (all the slot's columns lie in one kept run). Then every slot costs
// one shared-memory bit test: an untouched slot gets one 16-byte store of
// -inf (fp32 0xFF800000 or bf16 0xFF80 per column), a whole slot is skipped,
// and only the few slots at the edges of kept runs test their columns one by
// one (against a third bitmap, of candidate blocks).
#include "../../include/dsa_cb.h"

#include <cuda_runtime.h>

#include <cstdint>

#include "keys.cuh"

namespace dsa {
namespace {

// Columns per CTA: 32 KiB of logits (8192 fp32 or 16384 bf16 columns).
template <typename E>
__host__ __device__ constexpr int32_t mask_chunk() {
  return 32768 / E::kBytes;
}
constexpr int32_t kMaxMaskChunk = 16384;
constexpr int kMaskThreads = 256;
// A chunk's columns fall in at most 32768 / 16 + 1 aligned 16-byte slots
// (the chunk may start up to one slot minus an element past a boundary).
constexpr int32_t kSlots = 32768 / 16 + 1;
constexpr int32_t kSlotWords = (kSlots + 31) / 32;
// Blocks that overlap a chunk: at most its column count + 1 (block size 1).
constexpr int32_t kBlockBits = kMaxMaskChunk + 1;
constexpr int32_t kBlockWords = (kBlockBits + 31) / 32;

struct MaskArgs {
  void* logits;           // E::T elements
  int64_t ld;
  int64_t shard_stride;
  int32_t shards;         // 1: unsharded
  int64_t rows;
  int32_t width;          // (local) width
  const int32_t* row_ks;  // unsharded only, nullable
  const int32_t* row_ke;  // unsharded: ends; sharded: global ends
  int32_t row_repeat;
  int32_t block_size;     // (local) block
  const int32_t* cand;
  int32_t topk;
  int64_t ld_cand;
  int32_t chunks;         // chunks per row
};

template <typename E>
__device__ __forceinline__ void st_neg_inf16(typename E::T* p) {
  asm volatile("st.global.v4.b32 [%0], {%1, %1, %1, %1};" ::"l"(p), "r"(E::kNegInfWord)
               : "memory");
}
__device__ __forceinline__ void st_neg_inf1(float* p) { *p = neg_inf(); }
__device__ __forceinline__ void st_neg_inf1(uint16_t* p) { *p = 0xFF80u; }

// Sets bits [k0, k1) of a shared-memory bitmap (k0 < k1).
__device__ __forceinline__ void set_bits(uint32_t* bits, int32_t k0, int32_t k1) {
  const int32_t w0 = k0 >> 5, w1 = (k1 - 1) >> 5;
  for (int32_t w = w0; w <= w1; ++w) {
    const int32_t lo = w == w0 ? (k0 & 31) : 0;
    const int32_t hi = w == w1 ? ((k1 - 1) & 31) + 1 : 32;
    const uint32_t m = (hi == 32 ? ~0u : (1u << hi) - 1u) & ~((1u << lo) - 1u);
    atomicOr(bits + w, m);
  }
}

__device__ __forceinline__ bool test_bit(const uint32_t* bits, int32_t k) {
  return (bits[k >> 5] >> (k & 31)) & 1u;
}

template <typename E>
__global__ void __launch_bounds__(kMaskThreads) mask_kernel(const MaskArgs a) {
  constexpr int P = 16 / E::kBytes;  // columns per slot
  constexpr int kLogP = P == 4 ? 2 : 3;
  __shared__ uint32_t touch[kSlotWords];
  __shared__ uint32_t whole[kSlotWords];
  __shared__ uint32_t blocks[kBlockWords];
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
    // Shard d holds the global tokens t with t % shards == d: its window is
    // [ceil((gs - d) / shards), ceil((gke - d) / shards)), clamped to the
    // local width, with gs the clamped global start (0 without starts).
    const int32_t gke = __ldg(a.row_ke + g);
    const int32_t gs = a.row_ks ? min(max(__ldg(a.row_ks + g), 0), max(gke, 0)) : 0;
    auto local = [&](int32_t bound) -> int32_t {
      if (bound <= d) return 0;
      const uint32_t c = (static_cast<uint32_t>(bound - d) + static_cast<uint32_t>(a.shards - 1)) /
                         static_cast<uint32_t>(a.shards);
      return static_cast<int32_t>(min(c, static_cast<uint32_t>(a.width)));
    };
    e = local(gke);
    s = min(local(gs), e);
  }
  constexpr int32_t kChunk = mask_chunk<E>();
  const int32_t c0 = chunk * kChunk;
  const int32_t c1 = min(c0 + kChunk, a.width);
  typename E::T* rowp = static_cast<typename E::T*>(a.logits) +
                        static_cast<int64_t>(d) * a.shard_stride + row * a.ld;
  // 16-byte slots: slot k covers columns [a0 + P k, a0 + P k + P).
  const int32_t mis =
      static_cast<int32_t>((reinterpret_cast<uintptr_t>(rowp + c0) / E::kBytes) & (P - 1));
  const int32_t a0 = c0 - mis;
  const int32_t nslots = (c1 - a0 + P - 1) / P;  // <= kSlots

  for (int i = threadIdx.x; i < kSlotWords; i += kMaskThreads) {
    touch[i] = 0u;
    whole[i] = 0u;
  }
  // Only the words of the blocks that can overlap this chunk are used.
  const int32_t nbw = (kChunk / a.block_size + 2 + 31) / 32;
  for (int i = threadIdx.x; i < min(nbw, kBlockWords); i += kMaskThreads) blocks[i] = 0u;
  __syncthreads();

  // Kept columns of this chunk lie in [lo_c, hi_c), in blocks [blo, bhi).
  const int32_t lo_c = max(c0, s), hi_c = min(c1, e);
  const int32_t blo = lo_c < hi_c ? (lo_c - s) / a.block_size : 0;
  const int32_t bhi = lo_c < hi_c ? (hi_c - 1 - s) / a.block_size + 1 : 0;
  if (lo_c < hi_c) {
    const int32_t* crow = a.cand + row * a.ld_cand;
    for (int j = threadIdx.x; j < a.topk; j += kMaskThreads) {
      const int32_t b = __ldg(crow + j);
      if (b < blo || b >= bhi) continue;
      atomicOr(blocks + ((b - blo) >> 5), 1u << ((b - blo) & 31));
      // The kept run of block b inside the chunk (non-empty: b is in
      // [blo, bhi)).
      const int64_t bstart = static_cast<int64_t>(s) + static_cast<int64_t>(b) * a.block_size;
      const int32_t lo = static_cast<int32_t>(max(static_cast<int64_t>(lo_c), bstart));
      const int32_t hi =
          static_cast<int32_t>(min(static_cast<int64_t>(hi_c), bstart + a.block_size));
      set_bits(touch, (lo - a0) >> kLogP, ((hi - 1 - a0) >> kLogP) + 1);
      const int32_t f0 = (lo - a0 + P - 1) >> kLogP, f1 = (hi - a0) >> kLogP;
      if (f0 < f1) set_bits(whole, f0, f1);
    }
  }
  __syncthreads();

  for (int32_t k = threadIdx.x; k < nslots; k += kMaskThreads) {
    const int32_t cb = a0 + P * k;
    if (!test_bit(touch, k)) {
      if (cb >= c0 && cb + P <= c1) {
        st_neg_inf16<E>(rowp + cb);
      } else {
#pragma unroll
        for (int i = 0; i < P; ++i)
          if (cb + i >= c0 && cb + i < c1) st_neg_inf1(rowp + cb + i);
      }
      continue;
    }
    if (test_bit(whole, k)) continue;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int32_t c = cb + i;
      if (c < c0 || c >= c1) continue;
      const bool kept = c >= s && c < e && test_bit(blocks, (c - s) / a.block_size - blo);
      if (!kept) st_neg_inf1(rowp + c);
    }
  }
}

template <typename E>
dsa_status launch_mask(MaskArgs& a, cudaStream_t stream) {
  a.chunks = static_cast<int32_t>((static_cast<int64_t>(a.width) + mask_chunk<E>() - 1) /
                                  mask_chunk<E>());
  const int64_t grid = static_cast<int64_t>(a.shards) * a.rows * a.chunks;
  if (grid > INT32_MAX) return DSA_EUNSUPPORTED;
  mask_kernel<E><<<static_cast<unsigned>(grid), kMaskThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

template <typename E>
dsa_status mask_impl(typename E::T* logits, int64_t rows, int64_t width, int64_t ld_logits,
                     const int32_t* row_ks, const int32_t* row_ke, const int32_t* candidates,
                     int32_t topk_blocks, int64_t ld_candidates, int32_t block_size,
                     int32_t row_repeat, void* stream) {
  if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1 || topk_blocks < 0)
    return DSA_EINVAL;
  if (rows == 0 || width == 0) return DSA_OK;
  if (!logits || !row_ke || ld_logits < width) return DSA_EINVAL;
  if (topk_blocks > 0 && (!candidates || ld_candidates < topk_blocks)) return DSA_EINVAL;
  if (width > INT32_MAX - kMaxMaskChunk) return DSA_EUNSUPPORTED;
  MaskArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = 0;
  a.shards = 1;
  a.rows = rows;
  a.width = static_cast<int32_t>(width);
  a.row_ks = row_ks;
  a.row_ke = row_ke;
  a.row_repeat = row_repeat;
  a.block_size = block_size;
  a.cand = candidates;
  a.topk = topk_blocks;
  a.ld_cand = ld_candidates;
  return launch_mask<E>(a, static_cast<cudaStream_t>(stream));
}

template <typename E>
dsa_status mask_sharded_impl(typename E::T* logits, int32_t shards, int64_t rows,
                             int64_t local_width, int64_t ld_logits, int64_t shard_stride,
                             const int32_t* global_row_ks, const int32_t* global_row_ke,
                             int32_t global_block_size,
                             int32_t row_repeat, const int32_t* candidates, int32_t topk_blocks,
                             int64_t ld_candidates, void* stream) {
  if (shards < 1 || rows < 0 || local_width < 0 || global_block_size < 1 ||
      global_block_size % shards != 0 || row_repeat < 1 || topk_blocks < 0 ||
      ld_logits < local_width || shard_stride < 0)
    return DSA_EINVAL;
  if (rows == 0 || local_width == 0) return DSA_OK;
  if (!logits || !global_row_ke) return DSA_EINVAL;
  if (topk_blocks > 0 && (!candidates || ld_candidates < topk_blocks)) return DSA_EINVAL;
  if (local_width > INT32_MAX - kMaxMaskChunk) return DSA_EUNSUPPORTED;
  MaskArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = shard_stride;
  a.shards = shards;
  a.rows = rows;
  a.width = static_cast<int32_t>(local_width);
  a.row_ks = global_row_ks;
  a.row_ke = global_row_ke;
  a.row_repeat = row_repeat;
  a.block_size = global_block_size / shards;
  a.cand = candidates;
  a.topk = topk_blocks;
  a.ld_cand = ld_candidates;
  return launch_mask<E>(a, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_mask_candidate_logits(float* logits, int64_t rows, int64_t width,
                                                int64_t ld_logits, const int32_t* row_ks,
                                                const int32_t* row_ke, const int32_t* candidates,
                                                int32_t topk_blocks, int64_t ld_candidates,
                                                int32_t block_size, int32_t row_repeat,
                                                void* stream) {
  return dsa::mask_impl<dsa::F32>(logits, rows, width, ld_logits, row_ks, row_ke, candidates,
                                  topk_blocks, ld_candidates, block_size, row_repeat, stream);
}

extern "C" dsa_status dsa_mask_candidate_logits_bf16(uint16_t* logits, int64_t rows,
                                                     int64_t width, int64_t ld_logits,
                                                     const int32_t* row_ks,
                                                     const int32_t* row_ke,
                                                     const int32_t* candidates,
                                                     int32_t topk_blocks, int64_t ld_candidates,
                                                     int32_t block_size, int32_t row_repeat,
                                                     void* stream) {
  return dsa::mask_impl<dsa::BF16>(logits, rows, width, ld_logits, row_ks, row_ke, candidates,
                                   topk_blocks, ld_candidates, block_size, row_repeat, stream);
}

extern "C" dsa_status dsa_mask_candidate_logits_sharded(
    float* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ke, int32_t global_block_size,
    int32_t row_repeat, const int32_t* candidates, int32_t topk_blocks, int64_t ld_candidates,
    void* stream) {
  return dsa::mask_sharded_impl<dsa::F32>(logits, shards, rows, local_width, ld_logits,
                                          shard_stride, nullptr, global_row_ke, global_block_size,
                                          row_repeat, candidates, topk_blocks, ld_candidates,
                                          stream);
}

extern "C" dsa_status dsa_mask_candidate_logits_sharded_bf16(
    uint16_t* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ke, int32_t global_block_size,
    int32_t row_repeat, const int32_t* candidates, int32_t topk_blocks, int64_t ld_candidates,
    void* stream) {
  return dsa::mask_sharded_impl<dsa::BF16>(logits, shards, rows, local_width, ld_logits,
                                           shard_stride, nullptr, global_row_ke, global_block_size,
                                           row_repeat, candidates, topk_blocks, ld_candidates,
                                           stream);
}

extern "C" dsa_status dsa_mask_candidate_logits_sharded_starts(
    float* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ks, const int32_t* global_row_ke,
    int32_t global_block_size, int32_t row_repeat, const int32_t* candidates,
    int32_t topk_blocks, int64_t ld_candidates, void* stream) {
  return dsa::mask_sharded_impl<dsa::F32>(logits, shards, rows, local_width, ld_logits,
                                          shard_stride, global_row_ks, global_row_ke,
                                          global_block_size, row_repeat, candidates, topk_blocks,
                                          ld_candidates, stream);
}

extern "C" dsa_status dsa_mask_candidate_logits_sharded_starts_bf16(
    uint16_t* logits, int32_t shards, int64_t rows, int64_t local_width, int64_t ld_logits,
    int64_t shard_stride, const int32_t* global_row_ks, const int32_t* global_row_ke,
    int32_t global_block_size, int32_t row_repeat, const int32_t* candidates,
    int32_t topk_blocks, int64_t ld_candidates, void* stream) {
  return dsa::mask_sharded_impl<dsa::BF16>(logits, shards, rows, local_width, ld_logits,
                                           shard_stride, global_row_ks, global_row_ke,
                                           global_block_size, row_repeat, candidates,
                                           topk_blocks, ld_candidates, stream);
}
