// kvs_cluster.cuh -- stores into another block's shared memory within a
// thread-block cluster, and the split cluster barrier that makes them safe.
//
// A block may write another block's shared memory only once that block has
// started: every thread arrives (relaxed) at a cluster barrier on entry and
// waits on it before its first remote store.  The arrive costs nothing and
// the wait, far later, finds the barrier long complete.  Remote stores are
// visible to their target after the next full cluster barrier
// (barrier.cluster.arrive.release + wait.acquire).
#pragma once

#include <cstdint>

namespace kvs {

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait;" ::: "memory");
}

// a: an address from mapa (dsmem_addr)
__device__ __forceinline__ void st_dsmem_f4(uint32_t a, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_dsmem_f2(uint32_t a, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y)
               : "memory");
}

__device__ __forceinline__ void st_dsmem_f32(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem_s32(uint32_t a, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

}  // namespace kvs
