// bulk.cuh -- mbarrier and 1-D bulk-copy (cp.async.bulk) helpers for sm_103a.
//
// Every wait here is bounded: after about two seconds it gives up and returns
// false, so a kernel can flag the failure and finish instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr uint64_t kBulkWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t bulk_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Bounded wait for phase `parity` of an mbarrier; false if it gave up.  try_wait
// suspends the thread until the phase completes or a short system limit passes;
// the clock is read every 256 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = bulk_timer_ns();
  for (unsigned it = 1; !mbar_try_wait(bar, parity); ++it)
    if ((it & 255u) == 0 && bulk_timer_ns() - t0 > kBulkWaitNs) return false;
  return true;
}

// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// memory into shared memory, completing that many transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace nvfp4
