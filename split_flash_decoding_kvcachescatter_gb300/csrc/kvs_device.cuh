// kvs_device.cuh -- device-side building blocks for sm_103a: mbarrier
// waits with a wall-clock bound, 1-D bulk asynchronous copies (TMA,
// cp.async.bulk) global -> shared, and the status word.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvsdecode.h"

namespace kvs {

// Upper bound on any single pipeline wait.  A wait that runs past it means a
// bug (a copy that never lands, a role that died); the kernel then records
// KVS_ERR_TIMEOUT and returns instead of spinning forever.
constexpr uint64_t kWaitLimitNs = KVS_WAIT_LIMIT_DEFAULT_NS;  // 2 s

// The bound of the polling variant's waits (below): each translation unit
// with waits has its own copy, set on the current device by
// kvs_set_wait_limit_ns and read at run time.
static __constant__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

// Host: sets this translation unit's copy of the bound on the current device.
static inline cudaError_t set_unit_wait_limit(uint64_t ns) {
  const unsigned long long v = ns;
  return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v));
}

__device__ __forceinline__ void record_status(int *d_status, int code) {
  if (d_status != nullptr) atomicCAS(d_status, 0, code);
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible (a no-op when the kernel
// was launched without programmatic stream serialisation) ...
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// ... and let the next kernel in the stream start launching now.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// Potentially blocking test: the thread may be suspended for a while (until
// the phase completes or a hardware time limit passes).
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Returns false
// if *abort became non-zero or the wait ran past its bound.
//   kPoll = false (kernels launched at the default bound): the thread sleeps
//     in mbarrier.try_wait (the hardware wakes it when the phase completes,
//     or after about 4 us) and looks at the abort flag and the clock every
//     64 tries, against the fixed kWaitLimitNs.  Nothing is added to a wait
//     that finds its phase complete.
//   kPoll = true (kernels launched while kvs_set_wait_limit_ns has lowered
//     the bound, to test the timeout path): the thread polls with the
//     non-blocking test_wait and looks at the abort flag and the clock at
//     every poll, against g_wait_limit_ns, so a bound of 0 ends the first
//     wait that does not find its phase complete.
template <bool kPoll>
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile int *abort) {
  if (!kPoll) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((it & 63u) == 0) {
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
      }
    }
  }
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t limit = g_wait_limit_ns;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 >= limit) return false;
  }
}

// A drain wait: for work this block already issued (a bulk copy into its
// shared memory, tensor-core products) to finish before the block moves on
// or exits.  No abort flag, and always the full kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (evict_first for data read once).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

// ---- thread-block clusters ----------------------------------------------
// Every thread of every block of the cluster must execute it, on every path.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in cluster block `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ int ld_dsmem_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ float neg_inf_f() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

}  // namespace kvs
