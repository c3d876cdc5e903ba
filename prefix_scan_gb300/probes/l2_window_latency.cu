// l2_window_latency.cu -- what one look-back window's loads cost in L2.
//
// One warp makes dependent 32-lane loads (ld.relaxed.gpu, like the
// look-back's descriptor polls) of 64-byte-strided slots of a 2 MiB,
// L2-resident array: lane l reads slot (base + l), and the next base comes
// from lane 0's value, so each load waits for the one before.  The average
// time per load is the L2 round trip of one 32-descriptor window.  It runs
// alone, then again while every other SM streams a copy of 1 GiB at full
// rate (1 + 2 x SMs CTAs; CTA 0 holds the probing warp).  A measurement tool
// of the trace build's kind: it is not part of the library.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#define CHECK(x)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (x);                                                             \
        if (e_ != cudaSuccess) {                                                          \
            std::printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__);  \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__global__ void probe(const unsigned long long *slots, long long nslots, int stride_words, int iters,
                      const uint4 *src, uint4 *dst, long long nvec, int copy_reps, unsigned long long *out) {
    if (blockIdx.x == 0) {
        if (threadIdx.x >= 32) return;
        const int lane = threadIdx.x;
        unsigned long long base = 0;
        for (int it = 0; it < 64; ++it) {   // bring the slots into L2
            unsigned long long v;
            const unsigned long long *p = slots + ((base + lane) % nslots) * stride_words;
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
            base = __shfl_sync(0xffffffffu, v, 0);
        }
        const unsigned long long t_wait = now_ns();
        while (now_ns() - t_wait < 20000ull) {}   // let the copy reach full rate
        const unsigned long long t0 = now_ns();
        for (int it = 0; it < iters; ++it) {
            unsigned long long v;
            const unsigned long long *p = slots + ((base + lane) % nslots) * stride_words;
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
            base = __shfl_sync(0xffffffffu, v, 0);
        }
        const unsigned long long t1 = now_ns();
        if (lane == 0) {
            out[0] = t1 - t0;
            out[1] = base;   // keeps the chain live
        }
        return;
    }
    const long long nthreads = (long long)(gridDim.x - 1) * blockDim.x;
    const long long tid = (long long)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    for (int rep = 0; rep < copy_reps; ++rep)
        for (long long i = tid; i < nvec; i += nthreads) {
            uint4 v;
            asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(src + i));
            asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                         :: "l"(dst + i), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
        }
}

int main() {
    const long long nslots = 1 << 15;   // 32768 slots of 64 bytes: 2 MiB
    const int stride_words = 8;
    std::vector<unsigned long long> h((size_t)nslots * stride_words, 0);
    std::srand(1);
    // each slot names the next window's base: a multiple of 32 slots
    for (long long i = 0; i < nslots; ++i)
        h[(size_t)i * stride_words] = (unsigned long long)(std::rand() % (nslots / 32)) * 32;
    unsigned long long *slots = nullptr, *out = nullptr;
    CHECK(cudaMalloc(&slots, h.size() * sizeof(h[0])));
    CHECK(cudaMemcpy(slots, h.data(), h.size() * sizeof(h[0]), cudaMemcpyHostToDevice));
    CHECK(cudaMalloc(&out, 2 * sizeof(unsigned long long)));
    const long long nvec = (1ll << 30) / 16;   // 1 GiB copied, 16 times over
    uint4 *src = nullptr, *dst = nullptr;
    CHECK(cudaMalloc(&src, nvec * 16));
    CHECK(cudaMalloc(&dst, nvec * 16));
    CHECK(cudaMemset(src, 1, nvec * 16));
    int sms = 0;
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    const int iters = 2000;
    for (int loaded = 0; loaded < 2; ++loaded)
        for (int rep = 0; rep < 3; ++rep) {
            probe<<<loaded ? 1 + 2 * sms : 1, 512>>>(slots, nslots, stride_words, iters, src, dst, nvec, 16, out);
            CHECK(cudaGetLastError());
            CHECK(cudaDeviceSynchronize());
            unsigned long long o[2];
            CHECK(cudaMemcpy(o, out, sizeof(o), cudaMemcpyDeviceToHost));
            std::printf("%s: %.1f ns per dependent 32-lane window load\n", loaded ? "under a full-rate copy" : "idle",
                        (double)o[0] / iters);
        }
    CHECK(cudaFree(src));
    CHECK(cudaFree(dst));
    CHECK(cudaFree(slots));
    CHECK(cudaFree(out));
    return 0;
}
