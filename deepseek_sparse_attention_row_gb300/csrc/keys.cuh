// keys.cuh -- order-preserving uint32 keys for fp32 scores, the NaN-propagating
// max, and streaming global loads.
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

}  // namespace dsa
