// dcp_lse.cu -- the DCP partial-attention LSE correction and the merge over
// shards: the C ABI dsa_correct_attn_out / dsa_merge_attn_out of
// include/dsa_dcp_attn.h.
//
// sglang dcp/kernels.py, _correct_attn_cp_out_kernel and correct_attn_out.
// Each of N context shards computed attention over its own keys: a partial
// output o_n[b,h,:] and a base-2 log-sum-exp l_n[b,h]. Per (b, h):
//   x_n = l_n, with NaN and +inf read as -inf;
//   m   = max_n x_n, or 0 when every x_n is -inf;
//   F   = log2(sum_n 2^(x_n - m)) + m;
//   f_n = 2^(l_n - F), with a NaN or +inf exponent read as -inf (share 0).
// The correction writes F and f_i * o_i for one shard i, head-major
// ([H, B, Dh]) as on the page; the merge writes sum_n f_n * o_n, the
// cross-shard sum that follows the correction, for all N shards held on
// this GPU as a leading axis.
//
// Both are streaming passes bound by HBM bandwidth: one warp per (b, h) row
// at a time. Lane n < N loads l_n (adjacent warps take adjacent heads, so
// the LSE sectors are shared in L2), the warp reduces max and sum with
// shuffles, and the row's Dh values move in 16-byte vectors when the layout
// allows (unit stride, aligned rows), else one element per lane and step.
// All arithmetic is fp32; bf16 data is widened on load and rounded to
// nearest even on store.
#include "../../include/dsa_dcp_attn.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace dsa {
namespace {

constexpr int kLseThreads = 256;
constexpr int kLseWarps = kLseThreads / 32;
constexpr int32_t kMaxLseShards = 32;  // one lane per shard

struct LseArgs {
  const void* in;        // correction: o_i [B, H, Dh]; merge: o [N, B, H, Dh]
  int64_t in_sn, in_sb, in_sh, in_sd;
  const float* lses;     // [N, B, H]
  int64_t l_sn, l_sb, l_sh;
  int32_t shards;
  int32_t rank;          // correction only
  int64_t batch, heads;
  int32_t head_dim;
  void* out;             // [H, B, Dh]
  int64_t o_sh, o_sb, o_sd;
  float* lse_out;        // [B, H], nullable
  int64_t lo_sb, lo_sh;
};

__device__ __forceinline__ float neg_inf_f() { return __int_as_float(0xff800000); }

// NaN and +inf count as -inf.
__device__ __forceinline__ float clean(float x) {
  return (x != x || x == __int_as_float(0x7f800000)) ? neg_inf_f() : x;
}

// The combined LSE F of one (b, h) row; lane n < N also returns its raw
// l_n in `mine` (-inf on other lanes).
__device__ __forceinline__ float combined_lse(const LseArgs& a, int64_t b, int64_t h, float& mine) {
  const int lane = threadIdx.x & 31;
  mine = neg_inf_f();
  if (lane < a.shards) mine = __ldg(a.lses + lane * a.l_sn + b * a.l_sb + h * a.l_sh);
  const float x = clean(mine);
  float m = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (m == neg_inf_f()) m = 0.0f;
  float t = exp2f(x - m);  // 0 for x = -inf, and on lanes past N
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return log2f(t) + m;
}

// f = 2^(l - F), a NaN or +inf exponent giving 0.
__device__ __forceinline__ float share_of(float l, float F) {
  float dlt = l - F;
  if (dlt != dlt || dlt == __int_as_float(0x7f800000)) dlt = neg_inf_f();
  return exp2f(dlt);
}

template <typename T>
struct Vec;  // 16 bytes of T, widened to fp32
template <>
struct Vec<float> {
  static constexpr int kN = 4;
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ void store(float* p) const {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  float v[8];
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void narrow(float* p, float x) { *p = x; }
__device__ __forceinline__ void narrow(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// One warp per (b, h) row, rows in a grid-stride loop (h fastest).
// VEC: 16-byte vectors (unit stride in Dh, rows 16-byte aligned, Dh a
// multiple of the vector) or scalars.
template <typename T, bool VEC, bool MERGE>
__global__ void __launch_bounds__(kLseThreads) lse_kernel(const LseArgs a) {
  // Merge: the shares f_n of the warp's current row (lanes that leave the
  // element loop early cannot serve shuffles, so the loop reads them here).
  __shared__ float shares[kLseWarps][kMaxLseShards];
  float* f_row = shares[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int64_t nrows = a.batch * a.heads;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kLseWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kLseWarps;
  const T* in = static_cast<const T*>(a.in);
  T* out = static_cast<T*>(a.out);
  for (int64_t r = warp0; r < nrows; r += nwarps) {
    const int64_t b = r / a.heads, h = r % a.heads;
    float mine;
    const float F = combined_lse(a, b, h, mine);
    if (a.lse_out && lane == 0) a.lse_out[b * a.lo_sb + h * a.lo_sh] = F;
    // Correction: only shard `rank`'s share. Merge: lane n holds f_n.
    const float f_lane = share_of(mine, F);
    const float f_rank = MERGE ? 0.0f : __shfl_sync(0xffffffffu, f_lane, a.rank);
    if (MERGE) {
      __syncwarp();  // the previous row's shares have been read
      f_row[lane] = f_lane;
      __syncwarp();
    }
    const T* src = in + b * a.in_sb + h * a.in_sh;
    T* dst = out + h * a.o_sh + b * a.o_sb;
    if constexpr (VEC) {
      constexpr int kN = Vec<T>::kN;
      const int32_t nvec = a.head_dim / kN;
      for (int32_t j = lane; j < nvec; j += 32) {
        Vec<T> acc;
        if constexpr (MERGE) {
#pragma unroll
          for (int i = 0; i < kN; ++i) acc.v[i] = 0.0f;
          for (int32_t n = 0; n < a.shards; ++n) {
            const float fn = f_row[n];
            Vec<T> x;
            x.load(src + n * a.in_sn + static_cast<int64_t>(j) * kN);
#pragma unroll
            for (int i = 0; i < kN; ++i) acc.v[i] = fmaf(fn, x.v[i], acc.v[i]);
          }
        } else {
          acc.load(src + static_cast<int64_t>(j) * kN);
#pragma unroll
          for (int i = 0; i < kN; ++i) acc.v[i] *= f_rank;
        }
        acc.store(dst + static_cast<int64_t>(j) * kN);
      }
    } else {
      for (int32_t j = lane; j < a.head_dim; j += 32) {
        float acc;
        if constexpr (MERGE) {
          acc = 0.0f;
          for (int32_t n = 0; n < a.shards; ++n) {
            const float fn = f_row[n];
            acc = fmaf(fn, widen(src[n * a.in_sn + j * a.in_sd]), acc);
          }
        } else {
          acc = f_rank * widen(src[j * a.in_sd]);
        }
        narrow(dst + j * a.o_sd, acc);
      }
    }
  }
}

// Streaming multiprocessors of the current device, cached per device.
int sm_count_lse() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 152;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Resident CTAs per SM of one kernel instantiation on the current device
// (asked once per device).
template <typename T, bool VEC, bool MERGE>
int resident_ctas() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 4;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, lse_kernel<T, VEC, MERGE>, kLseThreads,
                                                      0) != cudaSuccess || n <= 0)
      return 4;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <typename T, bool VEC, bool MERGE>
dsa_status launch_lse_shape(const LseArgs& a, cudaStream_t stream) {
  const int64_t rows = a.batch * a.heads;
  const int64_t want = (rows + kLseWarps - 1) / kLseWarps;
  // One wave: every SM holds as many CTAs as fit, each CTA's warps then
  // stride over the rows (no partial second wave); fewer when rows are few.
  const int64_t cap = static_cast<int64_t>(sm_count_lse()) * resident_ctas<T, VEC, MERGE>();
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  lse_kernel<T, VEC, MERGE><<<grid, kLseThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

template <typename T, bool MERGE>
dsa_status launch_lse(const LseArgs& a, bool vec, cudaStream_t stream) {
  return vec ? launch_lse_shape<T, true, MERGE>(a, stream)
             : launch_lse_shape<T, false, MERGE>(a, stream);
}

// 16-byte vectors apply when Dh has unit stride, is a whole number of
// vectors, and every row start is 16-byte aligned (base and the B / H / N
// strides, in bytes, multiples of 16).
bool vec_ok(const LseArgs& a, size_t esize, bool merge) {
  const int64_t per = 16 / static_cast<int64_t>(esize);
  auto al = [&](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (a.in_sd != 1 || a.o_sd != 1 || a.head_dim % per != 0) return false;
  if (!al(a.in) || !al(a.out)) return false;
  if (a.in_sb % per || a.in_sh % per || (merge && a.in_sn % per)) return false;
  if (a.o_sb % per || a.o_sh % per) return false;
  return true;
}

dsa_status run_lse(LseArgs& a, int32_t dtype, bool merge, cudaStream_t stream) {
  if (dtype == DSA_DTYPE_F32) {
    const bool v = vec_ok(a, 4, merge);
    return merge ? launch_lse<float, true>(a, v, stream) : launch_lse<float, false>(a, v, stream);
  }
  const bool v = vec_ok(a, 2, merge);
  return merge ? launch_lse<__nv_bfloat16, true>(a, v, stream)
               : launch_lse<__nv_bfloat16, false>(a, v, stream);
}

bool bad_common(int32_t dtype, int32_t shards, int64_t batch, int64_t heads, int64_t head_dim) {
  return (dtype != DSA_DTYPE_F32 && dtype != DSA_DTYPE_BF16) || shards < 1 || batch < 0 ||
         heads < 0 || head_dim < 0;
}

}  // namespace
}  // namespace dsa

extern "C" int32_t dsa_attn_max_shards(void) { return dsa::kMaxLseShards; }

extern "C" dsa_status dsa_correct_attn_out(
    const void* out, int32_t dtype, int64_t batch, int64_t heads, int64_t head_dim,
    int64_t out_sb, int64_t out_sh, int64_t out_sd, const float* lses, int32_t shards,
    int64_t lse_sn, int64_t lse_sb, int64_t lse_sh, int32_t rank, void* new_out,
    int64_t new_sh, int64_t new_sb, int64_t new_sd, float* lse_out, int64_t lo_sb,
    int64_t lo_sh, void* stream) {
  if (dsa::bad_common(dtype, shards, batch, heads, head_dim) || rank < 0 || rank >= shards)
    return DSA_EINVAL;
  if (shards > dsa::kMaxLseShards || head_dim > INT32_MAX) return DSA_EUNSUPPORTED;
  if (batch == 0 || heads == 0) return DSA_OK;
  if (!lses || (head_dim > 0 && (!out || !new_out))) return DSA_EINVAL;
  dsa::LseArgs a{};
  a.in = out;
  a.in_sn = 0;
  a.in_sb = out_sb;
  a.in_sh = out_sh;
  a.in_sd = out_sd;
  a.lses = lses;
  a.l_sn = lse_sn;
  a.l_sb = lse_sb;
  a.l_sh = lse_sh;
  a.shards = shards;
  a.rank = rank;
  a.batch = batch;
  a.heads = heads;
  a.head_dim = static_cast<int32_t>(head_dim);
  a.out = new_out;
  a.o_sh = new_sh;
  a.o_sb = new_sb;
  a.o_sd = new_sd;
  a.lse_out = lse_out;
  a.lo_sb = lo_sb;
  a.lo_sh = lo_sh;
  return dsa::run_lse(a, dtype, false, static_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_merge_attn_out(
    const void* outs, int32_t dtype, int32_t shards, int64_t batch, int64_t heads,
    int64_t head_dim, int64_t outs_sn, int64_t outs_sb, int64_t outs_sh, int64_t outs_sd,
    const float* lses, int64_t lse_sn, int64_t lse_sb, int64_t lse_sh, void* merged,
    int64_t m_sh, int64_t m_sb, int64_t m_sd, float* lse_out, int64_t lo_sb, int64_t lo_sh,
    void* stream) {
  if (dsa::bad_common(dtype, shards, batch, heads, head_dim)) return DSA_EINVAL;
  if (shards > dsa::kMaxLseShards || head_dim > INT32_MAX) return DSA_EUNSUPPORTED;
  if (batch == 0 || heads == 0) return DSA_OK;
  if (!lses || (head_dim > 0 && (!outs || !merged))) return DSA_EINVAL;
  dsa::LseArgs a{};
  a.in = outs;
  a.in_sn = outs_sn;
  a.in_sb = outs_sb;
  a.in_sh = outs_sh;
  a.in_sd = outs_sd;
  a.lses = lses;
  a.l_sn = lse_sn;
  a.l_sb = lse_sb;
  a.l_sh = lse_sh;
  a.shards = shards;
  a.rank = 0;
  a.batch = batch;
  a.heads = heads;
  a.head_dim = static_cast<int32_t>(head_dim);
  a.out = merged;
  a.o_sh = m_sh;
  a.o_sb = m_sb;
  a.o_sd = m_sd;
  a.lse_out = lse_out;
  a.lo_sb = lo_sb;
  a.lo_sh = lo_sh;
  return dsa::run_lse(a, dtype, true, static_cast<cudaStream_t>(stream));
}
