// dsa_cb.cu -- sm_103a kernels and the C ABI of include/dsa_cb.h.
//
// One pass over HBM per call: every in-window logit is read once, block keys
// stay in shared memory, the top-k runs on them in place, and only ids (and,
// on request, block scores) are written back.
//
// Selecting kernel (select_kernel): one thread-block cluster of `csize` CTAs
// per row. The row's blocks that hold in-window data are split among the
// cluster's CTAs in units of 32 blocks; each CTA streams its share
// (stream.cuh) into its own shared-memory key array, then copies it into the
// leader CTA's array through distributed shared memory. After a cluster
// barrier the leader applies the pin, writes scores if asked, and runs the
// top-k (topk.cuh). Splitting long rows over a cluster keeps the largest unit
// of work small, so uneven row lengths do not leave SMs idle at the end.
// The DCP form is the same kernel reading `shards` slices per row and taking
// the max over them before the reduction, i.e. the all-reduce MAX of
// candidate_blocks.py's DCP branch happens in registers.
//
// Scores-only kernel (block_scores_kernel): one CTA per (row, chunk of
// blocks), no cluster, no top-k.
#include "../../include/dsa_cb.h"

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "keys.cuh"
#include "stream.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int32_t kMaxSelectBlocks = 16384;
constexpr int32_t kMaxShards = 1024;
constexpr int32_t kSplitUnit = 32;  // blocks per unit of the in-cluster split
constexpr int kMaxCluster = 8;

struct SelectArgs {
  const float* logits;
  int64_t ld;            // row stride (elements)
  int64_t shard_stride;  // sharded: elements between shards
  int32_t shards;        // 1 for the unsharded form
  int32_t width;         // unsharded width, or local width of each shard
  const int32_t* row_ks;  // unsharded only, nullable
  const int32_t* row_ke;  // unsharded: window ends; sharded: global ends
  int32_t row_repeat;
  int32_t block_size;    // unsharded block, or local block of each shard
  int32_t global_block_size;
  int32_t nb;            // blocks per output row
  int32_t nb_data;       // blocks that can hold data (sharded: min(ceil(lw/lbs), nbg))
  int32_t pin_newest;    // unsharded only
  int32_t topk;
  int32_t kpad;
  int32_t* out;
  int64_t ld_out;
  float* scores;
  int64_t ld_scores;
};

struct RowPlan {
  const float* origin;
  int32_t len_max;
  int32_t nblk;       // blocks holding in-window data
  int32_t pin_block;  // -1: none
  int vec, lpb_log2;
};

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Window of an unsharded row: e = min(ke, width), s = min(max(ks, 0), e).
// Every thread computes the same plan from the row's bounds.
__device__ __forceinline__ RowPlan plan_unsharded(const float* logits, int64_t ld, int32_t width,
                                                  const int32_t* row_ks, const int32_t* row_ke,
                                                  int32_t row_repeat, int32_t block_size,
                                                  int32_t pin_newest, int64_t row) {
  const int64_t g = row / row_repeat;
  const int32_t ks = row_ks ? __ldg(row_ks + g) : 0;
  const int32_t ke = __ldg(row_ke + g);
  const int32_t e = min(ke, width);
  const int32_t s = min(max(ks, 0), e);
  const uint32_t n = e > s ? static_cast<uint32_t>(e - s) : 0u;
  RowPlan p;
  p.origin = logits + row * ld + s;
  p.len_max = static_cast<int32_t>(n);
  p.nblk = static_cast<int32_t>((n + static_cast<uint32_t>(block_size) - 1u) /
                                static_cast<uint32_t>(block_size));
  p.pin_block = (pin_newest && n > 0) ? static_cast<int32_t>((n - 1u) / block_size) : -1;
  p.vec = choose_vec(p.origin, block_size, &p.lpb_log2);
  return p;
}

// Local end of shard d for global end gke: shard d holds the global tokens
// t = shards*c + d, so those below gke are its first ceil((gke - d) / shards)
// local columns; clamped to the local width.
__device__ __forceinline__ int32_t shard_len(int32_t gke, int32_t d, int32_t shards, int32_t lw) {
  if (gke <= d) return 0;
  const uint32_t lke = (static_cast<uint32_t>(gke - d) + static_cast<uint32_t>(shards - 1)) /
                       static_cast<uint32_t>(shards);
  return static_cast<int32_t>(min(lke, static_cast<uint32_t>(lw)));
}

template <int SVEC>
__device__ __forceinline__ void stream_sharded(const Window& w, int lpb_log2, int32_t block_size,
                                               int32_t b0, int32_t b1, uint32_t* keys) {
  if constexpr (SVEC == 4)
    stream_pow2<4, 1, 8>(w, lpb_log2, b0, b1, keys, 0);
  else if constexpr (SVEC == 2)
    stream_pow2<2, 2, 8>(w, lpb_log2, b0, b1, keys, 0);
  else if constexpr (SVEC == 1)
    stream_pow2<1, 4, 8>(w, lpb_log2, b0, b1, keys, 0);
  else
    stream_generic<4, 8>(w, block_size, b0, b1, keys, 0);
}

// One row per cluster of csize CTAs (csize is 1 unless overridden).
// SHARDED = false: unsharded rows, vector width chosen per row.
// SHARDED = true: DCP rows; SVEC is the vector width fixed by the host
// (0 = generic path).
template <bool SHARDED, int SVEC>
__global__ void __launch_bounds__(kThreads, 4) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw);  // [max(kpad, kRankMax)]
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + max(a.kpad, kRankMax));  // [nb]
  int32_t* len = reinterpret_cast<int32_t*>(keys + a.nb);                // [shards]
  __shared__ TopkShared tsh;

  const uint32_t csize = cluster_size();
  const uint32_t crank = cluster_rank();
  const int64_t row = blockIdx.x / csize;

  RowPlan plan;
  int32_t gke = 0;
  if constexpr (SHARDED) {
    gke = __ldg(a.row_ke + row / a.row_repeat);
    const int32_t n0 = shard_len(gke, 0, a.shards, a.width);
    plan.origin = a.logits + row * a.ld;
    plan.len_max = n0;
    plan.nblk = min(static_cast<int32_t>((static_cast<uint32_t>(n0) + a.block_size - 1u) /
                                         static_cast<uint32_t>(a.block_size)),
                    a.nb_data);
    plan.pin_block = gke >= 1 ? static_cast<int32_t>(min(
                                    static_cast<uint32_t>(gke - 1) / a.global_block_size,
                                    static_cast<uint32_t>(a.nb - 1)))
                              : -1;
    plan.vec = SVEC;
    plan.lpb_log2 = SVEC ? __ffs(a.block_size / (SVEC ? SVEC : 1)) - 1 : 0;
    for (int d = threadIdx.x; d < a.shards; d += blockDim.x)
      len[d] = shard_len(gke, d, a.shards, a.width);
  } else {
    plan = plan_unsharded(a.logits, a.ld, a.width, a.row_ks, a.row_ke, a.row_repeat,
                          a.block_size, a.pin_newest, row);
    if (threadIdx.x == 0) len[0] = plan.len_max;
  }

  const int32_t nblk = plan.nblk;
  const int32_t units = (nblk + kSplitUnit - 1) / kSplitUnit;
  const int32_t b0 = min(static_cast<int32_t>(crank * units / csize) * kSplitUnit, nblk);
  const int32_t b1 = min(static_cast<int32_t>((crank + 1) * units / csize) * kSplitUnit, nblk);

  for (int32_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) keys[b] = kKeyNegInf;
  if (crank == 0)
    for (int32_t b = nblk + threadIdx.x; b < a.nb; b += blockDim.x) keys[b] = kKeyNegInf;
  __syncthreads();
  if (csize > 1) cluster_arrive();  // phase 0: this CTA has started

  Window w;
  w.origin = plan.origin;
  w.shard_stride = a.shard_stride;
  w.shards = a.shards;
  w.len = len;
  w.len_max = plan.len_max;
  if (b0 < b1) {
    if constexpr (SHARDED)
      stream_sharded<SVEC>(w, plan.lpb_log2, a.block_size, b0, b1, keys);
    else
      stream_row(w, plan.vec, plan.lpb_log2, a.block_size, b0, b1, keys, 0);
  }
  __syncthreads();
  if constexpr (SHARDED) {
    if constexpr (SVEC > 1)
      for (int d = threadIdx.x; d < a.shards; d += blockDim.x)
        commit_partial(load_partial<SVEC>(plan.origin + d * a.shard_stride, len[d], a.block_size,
                                          b0, b1),
                       keys, 0);
  } else {
    if (threadIdx.x == 0)
      commit_partial(load_partial_row(w, plan.vec, a.block_size, b0, b1), keys, 0);
  }
  __syncthreads();

  if (csize > 1) {
    cluster_wait();  // every CTA of the cluster has started
    if (crank != 0 && b0 < b1) {
      namespace cg = cooperative_groups;
      uint32_t* leader = cg::this_cluster().map_shared_rank(keys, 0);
      for (int32_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) leader[b] = keys[b];
    }
    cluster_arrive();  // phase 1: shares delivered
    cluster_wait();
    if (crank != 0) return;
  }

  // Leader: pin, scores, selection.
  topk_store(keys, a.nb, min(a.topk, a.nb), plan.pin_block, cand, a.kpad,
             a.topk > 0 ? a.out + row * a.ld_out : nullptr, a.topk,
             a.scores ? a.scores + row * a.ld_scores : nullptr, tsh);
}

struct ScoresArgs {
  const float* logits;
  int64_t ld;
  int32_t width;
  const int32_t* row_ks;
  const int32_t* row_ke;
  int32_t row_repeat;
  int32_t block_size;
  int32_t nb;
  int32_t pin_newest;
  int32_t chunk;   // blocks per CTA
  int32_t chunks;  // CTAs per row
  float* scores;
  int64_t ld_scores;
};

__global__ void __launch_bounds__(kThreads, 4) block_scores_kernel(const ScoresArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);  // [chunk]
  __shared__ int32_t len[1];
  const int64_t row = blockIdx.x / a.chunks;
  const int32_t c0 = static_cast<int32_t>(blockIdx.x % a.chunks) * a.chunk;
  const int32_t c1 = min(c0 + a.chunk, a.nb);

  const RowPlan plan = plan_unsharded(a.logits, a.ld, a.width, a.row_ks, a.row_ke, a.row_repeat,
                                      a.block_size, a.pin_newest, row);
  if (threadIdx.x == 0) len[0] = plan.len_max;
  for (int32_t b = threadIdx.x; b < c1 - c0; b += blockDim.x) keys[b] = kKeyNegInf;
  __syncthreads();
  const int32_t b0 = min(c0, plan.nblk), b1 = min(c1, plan.nblk);
  Window w;
  w.origin = plan.origin;
  w.shard_stride = 0;
  w.shards = 1;
  w.len = len;
  w.len_max = plan.len_max;
  if (b0 < b1) stream_row(w, plan.vec, plan.lpb_log2, a.block_size, b0, b1, keys, c0);
  __syncthreads();
  if (threadIdx.x == 0)
    commit_partial(load_partial_row(w, plan.vec, a.block_size, b0, b1), keys, c0);
  __syncthreads();
  if (threadIdx.x == 0 && plan.pin_block >= c0 && plan.pin_block < c1)
    keys[plan.pin_block - c0] = kKeyPosInf;
  __syncthreads();
  float* srow = a.scores + row * a.ld_scores;
  for (int32_t b = c0 + threadIdx.x; b < c1; b += blockDim.x) srow[b] = key_score(keys[b - c0]);
}

__global__ void fill_minus_one_kernel(int32_t* out, int64_t rows, int32_t cols, int64_t ld) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x)
    out[(i / cols) * ld + (i % cols)] = -1;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int g_cluster_override = -1;  // DSA_CB_CLUSTER: 0 = automatic, 1..8 forced
std::once_flag g_env_once;

int cluster_override() {
  std::call_once(g_env_once, [] {
    const char* s = std::getenv("DSA_CB_CLUSTER");
    g_cluster_override = s ? std::atoi(s) : 0;
    if (g_cluster_override < 0 || g_cluster_override > kMaxCluster) g_cluster_override = 0;
  });
  return g_cluster_override;
}

int32_t next_pow2(int32_t x) {
  int32_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

// CTAs per row. One by default: splitting rows over thread-block clusters
// measured slower on every workload (a cluster needs all its CTA slots free
// in one GPC at once). DSA_CB_CLUSTER=2..8 forces a split for experiments.
int choose_cluster(int64_t /*max_row_bytes*/) {
  const int forced = cluster_override();
  return forced > 0 ? forced : 1;
}

// Opts a kernel in to `smem` bytes of dynamic shared memory on the current
// device (static plus dynamic shared memory above 48 KiB needs the opt-in).
// Remembers the largest size set per (kernel, device) so repeated launches
// make no runtime call.
struct SmemOptIn {
  const void* fn;
  int device;
  size_t bytes;
};
std::mutex g_smem_mu;
SmemOptIn g_smem_table[64];
int g_smem_used = 0;

template <typename K>
cudaError_t set_smem_attr(K kernel, size_t smem) {
  if (smem == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const void* fn = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (int i = 0; i < g_smem_used; ++i) {
    if (g_smem_table[i].fn == fn && g_smem_table[i].device == dev) {
      if (g_smem_table[i].bytes >= smem) return cudaSuccess;
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err == cudaSuccess) g_smem_table[i].bytes = smem;
      return err;
    }
  }
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err == cudaSuccess && g_smem_used < 64) g_smem_table[g_smem_used++] = {fn, dev, smem};
  return err;
}

template <typename K>
dsa_status launch_select(K kernel, const SelectArgs& a, int64_t rows, int csize, size_t smem,
                         cudaStream_t stream) {
  if (set_smem_attr(kernel, smem) != cudaSuccess) return DSA_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * csize));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a) == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

dsa_status fill_minus_one(int32_t* out, int64_t rows, int32_t cols, int64_t ld, cudaStream_t s) {
  if (rows == 0 || cols == 0) return DSA_OK;
  const int64_t total = rows * cols;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, 4096));
  fill_minus_one_kernel<<<grid, 256, 0, s>>>(out, rows, cols, ld);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

size_t select_smem(int32_t kpad, int32_t nb, int32_t shards) {
  return static_cast<size_t>(std::max(kpad, kRankMax)) * 8 + static_cast<size_t>(nb) * 4 +
         static_cast<size_t>(shards) * 4;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_EINVAL: return "invalid argument";
    case DSA_ECUDA: return "CUDA runtime or launch failure";
    case DSA_EUNSUPPORTED: return "beyond this build's limits";
    default: return "unknown status";
  }
}

int32_t dsa_select_max_blocks(void) { return kMaxSelectBlocks; }
int32_t dsa_select_max_shards(void) { return kMaxShards; }

dsa_status dsa_block_scores(const float* logits, int64_t rows, int64_t width, int64_t ld_logits,
                            const int32_t* row_ks, const int32_t* row_ke, int32_t block_size,
                            int32_t row_repeat, int32_t pin_newest, float* scores_out,
                            int64_t ld_scores, void* stream) {
  if (rows < 0 || width < 0 || block_size < 1 || row_repeat < 1) return DSA_EINVAL;
  if (rows == 0 || width == 0) return DSA_OK;
  if (!logits || !row_ke || !scores_out || ld_logits < width) return DSA_EINVAL;
  const int64_t nb = (width + block_size - 1) / block_size;
  if (ld_scores < nb) return DSA_EINVAL;
  if (width > INT32_MAX - 64) return DSA_EUNSUPPORTED;

  ScoresArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.width = static_cast<int32_t>(width);
  a.row_ks = row_ks;
  a.row_ke = row_ke;
  a.row_repeat = row_repeat;
  a.block_size = block_size;
  a.nb = static_cast<int32_t>(nb);
  a.pin_newest = pin_newest != 0;
  // About 64 KiB of logits per CTA, at least 32 blocks, at most 4096.
  int64_t chunk = (64 * 1024 / 4) / block_size;
  chunk = std::max<int64_t>(32, std::min<int64_t>(4096, chunk));
  chunk = std::min<int64_t>(chunk, nb);
  a.chunk = static_cast<int32_t>(chunk);
  a.chunks = static_cast<int32_t>((nb + chunk - 1) / chunk);
  a.scores = scores_out;
  a.ld_scores = ld_scores;
  const size_t smem = static_cast<size_t>(chunk) * 4;
  if (set_smem_attr(block_scores_kernel, smem) != cudaSuccess) return DSA_ECUDA;
  const int64_t grid = rows * a.chunks;
  if (grid > INT32_MAX) return DSA_EUNSUPPORTED;
  block_scores_kernel<<<static_cast<unsigned>(grid), kThreads, smem,
                        static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ECUDA;
}

dsa_status dsa_select_candidate_blocks(const float* logits, int64_t rows, int64_t width,
                                       int64_t ld_logits, const int32_t* row_ks,
                                       const int32_t* row_ke, int32_t topk_blocks,
                                       int32_t block_size, int32_t row_repeat,
                                       int32_t pin_newest, int32_t* out, int64_t ld_out,
                                       float* scores_out, int64_t ld_scores, void* stream) {
  if (rows < 0 || width < 0 || topk_blocks < 0 || block_size < 1 || row_repeat < 1)
    return DSA_EINVAL;
  if (rows == 0) return DSA_OK;
  if (topk_blocks > 0 && (!out || ld_out < topk_blocks)) return DSA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (width == 0) return fill_minus_one(out, rows, topk_blocks, ld_out, s);
  if (!logits || !row_ke || ld_logits < width) return DSA_EINVAL;
  const int64_t nb = (width + block_size - 1) / block_size;
  if (scores_out && ld_scores < nb) return DSA_EINVAL;
  if (topk_blocks == 0 && !scores_out) return DSA_OK;
  if (nb > kMaxSelectBlocks || width > INT32_MAX - 64) return DSA_EUNSUPPORTED;
  if (rows * kMaxCluster > INT32_MAX) return DSA_EUNSUPPORTED;

  SelectArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = 0;
  a.shards = 1;
  a.width = static_cast<int32_t>(width);
  a.row_ks = row_ks;
  a.row_ke = row_ke;
  a.row_repeat = row_repeat;
  a.block_size = block_size;
  a.nb = static_cast<int32_t>(nb);
  a.nb_data = a.nb;
  a.pin_newest = pin_newest != 0;
  a.topk = topk_blocks;
  a.kpad = next_pow2(std::max<int32_t>(1, std::min<int32_t>(topk_blocks, a.nb)));
  a.out = out;
  a.ld_out = ld_out;
  a.scores = scores_out;
  a.ld_scores = ld_scores;
  const int csize = choose_cluster(width * 4);
  return launch_select(select_kernel<false, 0>, a, rows, csize, select_smem(a.kpad, a.nb, 1), s);
}

dsa_status dsa_select_candidate_blocks_sharded(const float* logits, int32_t shards, int64_t rows,
                                               int64_t local_width, int64_t ld_logits,
                                               int64_t shard_stride,
                                               const int32_t* global_row_ke,
                                               int32_t global_block_size,
                                               int32_t max_global_blocks, int32_t row_repeat,
                                               int32_t topk_blocks, int32_t* out, int64_t ld_out,
                                               float* scores_out, int64_t ld_scores,
                                               void* stream) {
  if (shards < 1 || rows < 0 || local_width < 0 || topk_blocks < 0 || global_block_size < 1 ||
      global_block_size % shards != 0 || row_repeat < 1 || ld_logits < local_width ||
      shard_stride < 0)
    return DSA_EINVAL;
  if (rows == 0) return DSA_OK;
  if (!global_row_ke || (topk_blocks > 0 && (!out || ld_out < topk_blocks))) return DSA_EINVAL;
  if (local_width > 0 && !logits) return DSA_EINVAL;
  const int32_t nbg = std::max<int32_t>(max_global_blocks, 1);
  if (scores_out && ld_scores < nbg) return DSA_EINVAL;
  if (topk_blocks == 0 && !scores_out) return DSA_OK;
  if (nbg > kMaxSelectBlocks || shards > kMaxShards || local_width > INT32_MAX - 64)
    return DSA_EUNSUPPORTED;
  if (rows * kMaxCluster > INT32_MAX) return DSA_EUNSUPPORTED;

  const int32_t lbs = global_block_size / shards;
  SelectArgs a{};
  a.logits = logits;
  a.ld = ld_logits;
  a.shard_stride = shard_stride;
  a.shards = shards;
  a.width = static_cast<int32_t>(local_width);
  a.row_ks = nullptr;
  a.row_ke = global_row_ke;
  a.row_repeat = row_repeat;
  a.block_size = lbs;
  a.global_block_size = global_block_size;
  a.nb = nbg;
  a.nb_data = static_cast<int32_t>(std::min<int64_t>((local_width + lbs - 1) / lbs, nbg));
  a.pin_newest = 0;
  a.topk = topk_blocks;
  a.kpad = next_pow2(std::max<int32_t>(1, std::min<int32_t>(topk_blocks, nbg)));
  a.out = out;
  a.ld_out = ld_out;
  a.scores = scores_out;
  a.ld_scores = ld_scores;

  // One vector width for every shard row: all shard origins must share the
  // alignment and the local block must split into a power of two of vectors.
  auto pow2 = [](int32_t x) { return x > 0 && (x & (x - 1)) == 0; };
  const uintptr_t base = reinterpret_cast<uintptr_t>(logits);
  auto aligned = [&](int vec) {
    return lbs % vec == 0 && pow2(lbs / vec) && (base % (4 * vec)) == 0 && ld_logits % vec == 0 &&
           shard_stride % vec == 0;
  };
  const size_t smem = select_smem(a.kpad, a.nb, shards);
  const int csize = choose_cluster(local_width * 4 * shards);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (aligned(4)) return launch_select(select_kernel<true, 4>, a, rows, csize, smem, s);
  if (aligned(2)) return launch_select(select_kernel<true, 2>, a, rows, csize, smem, s);
  if (pow2(lbs)) return launch_select(select_kernel<true, 1>, a, rows, csize, smem, s);
  return launch_select(select_kernel<true, 0>, a, rows, csize, smem, s);
}

}  // extern "C"
