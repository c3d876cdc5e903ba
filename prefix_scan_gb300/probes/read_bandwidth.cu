// read_bandwidth.cu -- how fast 1 GiB can be read from HBM, by the two routes
// the kernels use.
//
// (a) Plain 16-byte loads, grid-stride, four in flight per thread.
// (b) Bulk copies (cp.async.bulk) of one tile at a time into a ring of S
//     shared-memory stages per CTA, as the persistent kernels' producers do:
//     a producer thread fills a stage once the consumer warp hands it back,
//     and the consumer takes one word of each tile.  Tiles are assigned
//     statically (tile t to CTA t mod grid), so no claim or look-back is
//     involved: this is the read side of the pipeline alone.  The "halo"
//     rows copy 16 bytes before each tile as well, unaligned to 128 bytes,
//     as the run-length and reduce-by-key producers do.
// A device-to-device copy of the same bytes is timed for comparison (its
// line counts the bytes read only; the copy moves twice as many).  Every
// wait is bounded (one second by %globaltimer) and reported.  A measurement
// tool of the trace build's kind: it is not part of the library.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>

#define CHECK(x)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (x);                                                             \
        if (e_ != cudaSuccess) {                                                          \
            std::printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            std::exit(1);                                                                 \
        }                                                                                 \
    } while (0)

namespace {

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void bar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ void bar_expect(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_addr(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// false after a second without the phase
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity, unsigned long long t0) {
    while (!bar_try(b, parity))
        if (now_ns() - t0 > 1000000000ull) return false;
    return true;
}

__global__ void read_loads(const uint4 *src, long long nvec, unsigned *sink) {
    const long long nth = (long long)gridDim.x * blockDim.x;
    unsigned acc = 0;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * nth < nvec; i += 4 * nth) {
        const uint4 a = src[i], b = src[i + nth], c = src[i + 2 * nth], d = src[i + 3 * nth];
        acc ^= a.x ^ b.y ^ c.z ^ d.w;
    }
    for (; i < nvec; i += nth) acc ^= src[i].x;
    if (acc == 0x12345678u) sink[0] = acc;   // never true for the fill used; keeps the loads
}

// thread 0: producer; warp 1: consumer.  Stage s holds [16-byte halo][tile].
__global__ void read_bulk(const unsigned char *src, long long tiles, uint32_t tile_bytes, int stages, int halo,
                          unsigned *sink, int *err) {
    extern __shared__ __align__(128) unsigned char sm[];
    const uint32_t stage_bytes = tile_bytes + 16u;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)stages * stage_bytes);
    uint64_t *empty = full + stages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const unsigned long long t0 = now_ns();
    const long long mine = tiles > (long long)blockIdx.x ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (long long k = 0; k < mine; ++k) {
            const int s = (int)(k % stages);
            if (k >= stages && !bar_wait(&empty[s], (uint32_t)((k / stages - 1) & 1), t0)) {
                atomicExch(err, 1);
                break;
            }
            const long long t = blockIdx.x + k * gridDim.x;
            const uint32_t h = (halo && t > 0) ? 16u : 0u;   // tile 0 has nothing before it
            bar_expect(&full[s], tile_bytes + h);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(sm + (size_t)s * stage_bytes + 16u - h)),
                "l"(src + t * (long long)tile_bytes - h), "r"(tile_bytes + h), "r"(smem_addr(&full[s]))
                : "memory");
        }
    } else if (threadIdx.x >= 32 && threadIdx.x < 64) {
        const int lane = threadIdx.x & 31;
        unsigned acc = 0;
        for (long long k = 0; k < mine; ++k) {
            const int s = (int)(k % stages);
            if (!bar_wait(&full[s], (uint32_t)((k / stages) & 1), t0)) {
                atomicExch(err, 2);
                break;
            }
            acc ^= reinterpret_cast<const uint4 *>(sm + (size_t)s * stage_bytes + 16u)[lane].x;
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[s]);
        }
        if (acc == 0x12345678u) sink[1] = acc;
    }
}

}  // namespace

int main() {
    const long long bytes = 1ll << 30;
    unsigned char *src = nullptr, *dst = nullptr;
    unsigned *sink = nullptr;
    int *err = nullptr;
    CHECK(cudaMalloc(&src, bytes));
    CHECK(cudaMalloc(&dst, bytes));
    CHECK(cudaMalloc(&sink, 64));
    CHECK(cudaMalloc(&err, sizeof(int)));
    CHECK(cudaMemset(src, 1, bytes));
    CHECK(cudaMemset(err, 0, sizeof(int)));
    int sms = 0;
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    auto time_it = [&](const char *name, auto launch) {
        for (int i = 0; i < 3; ++i) launch();
        CHECK(cudaGetLastError());
        CHECK(cudaDeviceSynchronize());
        const int reps = 10;
        float best = 1e9f, sum = 0.f;
        for (int i = 0; i < reps; ++i) {
            CHECK(cudaEventRecord(e0));
            launch();
            CHECK(cudaEventRecord(e1));
            CHECK(cudaEventSynchronize(e1));
            float ms = 0.f;
            CHECK(cudaEventElapsedTime(&ms, e0, e1));
            best = ms < best ? ms : best;
            sum += ms;
        }
        int bad = 0;
        CHECK(cudaMemcpy(&bad, err, sizeof(int), cudaMemcpyDeviceToHost));
        std::printf("%-52s best %7.1f us %6.0f GB/s, mean %7.1f us %6.0f GB/s%s\n", name, best * 1e3,
                    bytes / (best * 1e-3) / 1e9, sum / reps * 1e3, bytes / (sum / reps * 1e-3) / 1e9,
                    bad ? "  (a wait gave up)" : "");
    };
    time_it("device-to-device copy (bytes read)", [&] {
        CHECK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice));
    });
    time_it("16-byte loads, 2 CTAs of 512 per SM", [&] {
        read_loads<<<sms * 2, 512>>>(reinterpret_cast<const uint4 *>(src), bytes / 16, sink);
    });
    struct Config {
        uint32_t tile_bytes;
        int stages, ctas_per_sm, halo;
    };
    const Config configs[] = {{32768, 3, 2, 0}, {32768, 3, 2, 1}, {32768, 2, 2, 0}, {32768, 2, 2, 1},
                              {65536, 3, 1, 0}, {16384, 6, 2, 0}, {16384, 3, 2, 0}};
    for (const Config &c : configs) {
        const size_t smem = (size_t)c.stages * (c.tile_bytes + 16) + 2 * (size_t)c.stages * 8;
        CHECK(cudaFuncSetAttribute(read_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        const long long tiles = bytes / c.tile_bytes;
        char name[96];
        std::snprintf(name, sizeof name, "bulk copies, %2u KiB x %d stages, %d CTA/SM%s", c.tile_bytes / 1024,
                      c.stages, c.ctas_per_sm, c.halo ? ", 16 B halo" : "");
        time_it(name, [&] {
            read_bulk<<<sms * c.ctas_per_sm, 64, smem>>>(src, tiles, c.tile_bytes, c.stages, c.halo, sink, err);
        });
    }
    return 0;
}
