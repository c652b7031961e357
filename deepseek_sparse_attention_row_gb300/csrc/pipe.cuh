// pipe.cuh -- shared-memory staging with the Blackwell bulk-copy engine:
// mbarriers, bounded waits, and cp.async.bulk (global -> shared) in inline PTX.
//
// A stage of a ring is filled by one cp.async.bulk per contiguous piece of
// global memory (16-byte aligned source, destination and size), counted on
// the stage's "full" mbarrier as transaction bytes; consumers wait on that
// barrier's phase and release the stage on its "empty" barrier. Every wait
// is bounded: after kWaitLimitNs of global time the waiter records the
// failure in a device-wide flag (pipe_error) and gives up, so that a bug in
// the byte accounting ends the kernel with an error the host can read
// instead of hanging the GPU.
#pragma once

#include <cstdint>

namespace dsa {

// Set (to the failing wait's site code) by a wait that timed out; read and
// cleared by the host through dsa_pipeline_error(). One copy per translation
// unit that includes this header (select_pipe.cu alone does).
static __device__ unsigned int g_pipe_error = 0u;

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes initialised mbarriers visible to the bulk-copy engine (async proxy).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One arrival plus `bytes` of expected transaction count for this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// One test of the phase. The thread may be suspended (up to kSuspendHintNs)
// until the phase completes, so that a waiting warp does not spin on issue
// slots that the folding and ranking warps need.
constexpr uint32_t kSuspendHintNs = 1000000u;  // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed. Returns false
// (after recording `site` in g_pipe_error) if that takes longer than
// kWaitLimitNs. Every waiter decides on its own clock only: warps that wait
// on the same phase then all see it complete, or all give up, and none is
// left alone at a barrier that its siblings have abandoned.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned site) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_pipe_error, 0u, site);
      return false;
    }
  }
}

// cp.async.bulk global -> shared: `bytes` (a multiple of 16) from the
// 16-byte aligned global address `src` to the 16-byte aligned shared address
// `dst`, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

}  // namespace dsa
