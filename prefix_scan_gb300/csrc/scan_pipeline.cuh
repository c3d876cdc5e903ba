// scan_pipeline.cuh -- shared-memory pipeline primitives for the
// persistent kernels: mbarriers (init, arrive, arrive with an expected
// byte count, bounded parity wait), the bulk asynchronous global-to-shared
// copy that completes on an mbarrier, and named barriers.  All inline PTX.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace ps {

constexpr uint32_t kMbarSpinCap = 1u << 22;   // try_wait rounds before giving up

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// try_wait with a suspend-time hint: the thread may be suspended until the
// phase completes or about `ns` nanoseconds have passed, instead of polling.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}
// Bounded wait that sleeps in the barrier: tries of up to `ns` nanoseconds
// each, for at most kMbarSpinCap tries or about two seconds, whichever ends
// first; false if it ran out.
constexpr unsigned long long kMbarWaitLimitNs = 2000000000ull;
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t *bar, uint32_t parity, uint32_t ns) {
    if (mbar_try_wait_for(bar, parity, ns)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0; i < kMbarSpinCap; ++i) {
        if (mbar_try_wait_for(bar, parity, ns)) return true;
        if ((i & 15u) == 15u && global_ns() - t0 > kMbarWaitLimitNs) return false;
    }
    return false;
}

// Bounded wait for the phase with the given parity; false if it ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kMbarSpinCap; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// The same for warps whose waits are long and off the critical path: after
// a few tries each retry sleeps `ns` nanoseconds, so the waiting warp stops
// taking issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_wait_sleepy(uint64_t *bar, uint32_t parity, uint32_t ns) {
    for (uint32_t i = 0; i < kMbarSpinCap; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 2) __nanosleep(ns);
    }
    return false;
}
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// A hint: fetch [src, src + bytes) from global memory into L2 (both 16-byte
// multiples / aligned); no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src_gmem), "r"(bytes) : "memory");
}
// A hint: fetch the line holding p into L2, to be evicted last.
__device__ __forceinline__ void prefetch_line_l2_last(const void *p) {
    asm volatile("prefetch.global.L2::evict_last [%0];" :: "l"(p) : "memory");
}
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// The compute warps of a CTA meet at a named barrier once per tile.  A warp
// whose bounded wait for its tile ran out must not leave the others waiting
// there: it raises the CTA's abort flag and meets them one last time; after
// that barrier every warp reads the flag and leaves the loop with it.
__device__ __forceinline__ void abort_meet(volatile int *flag, int id, int threads) {
    *flag = 1;
    named_barrier(id, threads);
}
__device__ __forceinline__ bool aborted(const volatile int *flag) { return *flag != 0; }

}  // namespace ps
