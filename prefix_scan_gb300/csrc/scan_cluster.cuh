// scan_cluster.cuh -- thread-block-cluster primitives (inline PTX) for the
// paired select kernel: this CTA's rank, addresses in the partner CTA's
// shared memory, stores there, arrivals on its mbarriers, a bounded wait
// that acquires at cluster scope, and the cluster barrier.
#pragma once

#include "scan_pipeline.cuh"

namespace ps {

// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared-memory address, in CTA `rank` of the cluster, of the variable
// that sits at `p` in this CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}
// Arrival on an mbarrier of another CTA of the cluster; it releases this
// thread's earlier writes (to that CTA's shared memory too) at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(addr) : "memory");
}
// Bounded wait on a local mbarrier that another CTA of the cluster arrives
// on: acquire at cluster scope, so that what that CTA wrote before arriving
// is visible; false if it ran out.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kMbarSpinCap; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
        if (ok) return true;
    }
    return false;
}
// Every thread of the cluster's CTAs meets here; memory operations before it
// are visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace ps
