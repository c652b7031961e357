// keys.cuh -- order-preserving uint32 keys for fp32 scores, the NaN-propagating
// max, streaming global loads, and the fp32 / bf16 element types.
//
// Block maxima and ranking both use one total order on fp32 values:
//   -inf < negative finite < -0 < +0 < positive finite < +inf < NaN,
// with every NaN equal. Mapping a value to the key
//   key(x) = x has its sign bit set ? ~bits(x) : bits(x) | 0x80000000
// makes unsigned integer order equal that order for non-NaN values, and
// every NaN is sent to the key of the canonical quiet NaN 0x7FC00000, which
// lies above the key of +inf. So a ranked top-k is a descending sort of keys,
// and results never depend on operand order (+0 / -0) or NaN payloads.
//
// Inside the streaming loop the max is taken on the floats themselves with
// PTX max.NaN.f32 (two or three operands): it returns a NaN whenever an
// operand is NaN and orders -0 below +0, i.e. it is the max of the total
// order above (the NaN-propagating max of candidate_blocks.py's
// _max_with_nan). Its NaN result is mapped to the canonical key when the
// accumulated value becomes a key.
#pragma once

#include <cstdint>

namespace dsa {

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // key(-inf): smallest key
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // key(+inf)
constexpr uint32_t kKeyNaN = 0xFFC00000u;     // key(canonical NaN): largest

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t k = b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
  return (x != x) ? kKeyNaN : k;
}

// Inverse of order_key on its image (NaN keys come back as 0x7FC00000).
__device__ __forceinline__ float key_score(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(b);
}

__device__ __forceinline__ float neg_inf() { return __uint_as_float(0xFF800000u); }

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float max_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed bf16 pairs: PTX max.NaN.bf16x2 takes the max of each 16-bit half
// separately; checked on GB300 to order every pair of special values (signed
// zeros, infinities, subnormals, NaNs of either sign) as the total order
// above in both halves, with a NaN result whenever an operand is NaN.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Read-only streaming loads: each logit is read once per call, so skip L1
// allocation.
__device__ __forceinline__ void ld_stream(const float* p, float (&x)[4]) {
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3])
      : "l"(p));
}
__device__ __forceinline__ void ld_stream(const float* p, float (&x)[2]) {
  asm("ld.global.nc.L1::no_allocate.v2.f32 {%0, %1}, [%2];"
      : "=f"(x[0]), "=f"(x[1])
      : "l"(p));
}
__device__ __forceinline__ void ld_stream(const float* p, float (&x)[1]) {
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(x[0]) : "l"(p));
}
__device__ __forceinline__ float ld_stream1(const float* p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Fold a vector into an accumulator with the NaN-propagating max.
__device__ __forceinline__ float fold(float acc, const float (&x)[4]) {
  return max_nan(max_nan(acc, x[0], x[1]), x[2], x[3]);
}
__device__ __forceinline__ float fold(float acc, const float (&x)[2]) {
  return max_nan(acc, x[0], x[1]);
}
__device__ __forceinline__ float fold(float acc, const float (&x)[1]) { return max_nan(acc, x[0]); }

// ---------------------------------------------------------------------------
// Element types of the logits
// ---------------------------------------------------------------------------
//
// F32: fp32 logits and scores. BF16: bf16 logits held as their 16-bit
// patterns; a bf16 value widens exactly to the fp32 value with those bits on
// top, so the max and the keys above apply unchanged to the widened values,
// and a bf16 score is the upper half of the fp32 score (exact: a block max
// is one of the block's values, +-inf, or the canonical NaN 0x7FC00000,
// whose upper half is the bf16 canonical NaN 0x7FC0).
struct F32 {
  using T = float;
  static constexpr int kBytes = 4;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;  // one -inf
};
struct BF16 {
  using T = uint16_t;
  static constexpr int kBytes = 2;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;  // two -inf
};

// VEC elements as loaded: whole 32-bit words (a lone bf16 sits in the low
// half of its word).
template <typename E, int VEC>
struct Raw {
  static constexpr int kWords = (VEC * E::kBytes + 3) / 4;
  uint32_t w[kWords];
};

template <typename E, int VEC>
__device__ __forceinline__ void raw_neg_inf(Raw<E, VEC>& r) {
#pragma unroll
  for (int i = 0; i < Raw<E, VEC>::kWords; ++i)
    r.w[i] = (E::kBytes * VEC >= 4) ? E::kNegInfWord : (E::kNegInfWord & 0xFFFFu);
}

// Streaming load of VEC elements (16, 8, 4 or 2 bytes, naturally aligned).
template <typename E, int VEC>
__device__ __forceinline__ void ld_raw(const typename E::T* p, Raw<E, VEC>& r) {
  constexpr int kB = VEC * E::kBytes;
  if constexpr (kB == 16) {
    asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
        : "l"(p));
  } else if constexpr (kB == 8) {
    asm("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
  } else if constexpr (kB == 4) {
    asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
  } else {
    static_assert(kB == 2, "vector of 2, 4, 8 or 16 bytes");
    r.w[0] = __ldg(reinterpret_cast<const unsigned short*>(p));
  }
}

// Element i of a loaded vector, widened to fp32.
template <typename E, int VEC>
__device__ __forceinline__ float raw_elem(const Raw<E, VEC>& r, int i) {
  if constexpr (E::kBytes == 4) {
    return __uint_as_float(r.w[i]);
  } else {
    const uint32_t w = r.w[i >> 1];
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
}

// Element r of a loaded 16-byte vector, r a runtime index (0 .. VEC-1),
// widened to fp32; selects on the bits of r, no local memory.
template <typename E, int VEC>
__device__ __forceinline__ float raw_elem_at(const Raw<E, VEC>& x, int r) {
  static_assert(VEC * E::kBytes == 16, "16-byte vectors");
  const int wi = E::kBytes == 4 ? r : (r >> 1);  // word holding element r
  const uint32_t lo2 = (wi & 1) ? x.w[1] : x.w[0];
  const uint32_t hi2 = (wi & 1) ? x.w[3] : x.w[2];
  const uint32_t w = (wi & 2) ? hi2 : lo2;
  if constexpr (E::kBytes == 4) return __uint_as_float(w);
  else return __uint_as_float((r & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Fold a loaded vector into an accumulator with the NaN-propagating max.
template <typename E, int VEC>
__device__ __forceinline__ float fold(float acc, const Raw<E, VEC>& r) {
  if constexpr (E::kBytes == 4) {
    float x[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) x[i] = __uint_as_float(r.w[i]);
    return fold(acc, x);
  } else if constexpr (VEC == 1) {
    return max_nan(acc, __uint_as_float(r.w[0] << 16));
  } else {
#pragma unroll
    for (int i = 0; i < Raw<E, VEC>::kWords; ++i)
      acc = max_nan(acc, __uint_as_float(r.w[i] << 16), __uint_as_float(r.w[i] & 0xFFFF0000u));
    return acc;
  }
}

// Element-wise NaN-propagating max of two loaded vectors, into a.
template <typename E, int VEC>
__device__ __forceinline__ void raw_max(Raw<E, VEC>& a, const Raw<E, VEC>& b) {
#pragma unroll
  for (int i = 0; i < Raw<E, VEC>::kWords; ++i) {
    if constexpr (E::kBytes == 4)
      a.w[i] = __float_as_uint(max_nan(__uint_as_float(a.w[i]), __uint_as_float(b.w[i])));
    else
      a.w[i] = max_nan_bf16x2(a.w[i], b.w[i]);
  }
}

// One element, widened (streaming scalar load).
__device__ __forceinline__ float ld_elem(const float* p) { return ld_stream1(p); }
__device__ __forceinline__ float ld_elem(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)))
                         << 16);
}

// A score written from its key, in the logits' type.
__device__ __forceinline__ void put_score(float* p, uint32_t key) { *p = key_score(key); }
__device__ __forceinline__ void put_score(uint16_t* p, uint32_t key) {
  *p = static_cast<uint16_t>(__float_as_uint(key_score(key)) >> 16);
}

}  // namespace dsa
