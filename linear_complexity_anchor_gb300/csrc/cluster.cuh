// Inline-PTX wrappers for thread-block clusters: CTA rank, distributed shared memory addresses
// and loads, mbarrier arrivals on another CTA's barrier and cluster-scope waits.
#pragma once

#include <stdint.h>

namespace anchor {
namespace cl {

__device__ __forceinline__ uint32_t ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// the address of this CTA's shared-memory location `addr` in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// (volatile, so they stay after the barrier wait that precedes them, but without a memory
// clobber, so that several can be in flight at once)
__device__ __forceinline__ float4 ld_f4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr));
    return v;
}

__device__ __forceinline__ float ld_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr));
    return v;
}

// one arrival on the mbarrier at `cluster_addr` (any CTA of the cluster), releasing this
// thread's earlier writes to the cluster
__device__ __forceinline__ void arrive_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// a non-blocking test of this CTA's mbarrier phase that acquires what the arriving threads of
// the cluster released
__device__ __forceinline__ bool test_wait_acquire(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// every thread of every CTA of the cluster: the barrier initialisations before it are visible
// to the whole cluster after it
__device__ __forceinline__ void sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace cl
}  // namespace anchor
