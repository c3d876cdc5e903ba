// host_link.cu -- how fast data crosses between pinned host memory and the
// GPU: 1 GiB each way by the copy engines (cudaMemcpyAsync, one direction,
// then both at once on two streams) and by kernels that read or write the
// pinned memory directly (plain 16-byte loads and stores through its device
// view, no bulk copies).  The end-to-end scan (ps_scan_host) can go no
// faster than the both-directions figure.  A measurement tool of the trace
// build's kind: it is not part of the library.
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("err %s line %d\n", cudaGetErrorString(e), __LINE__); exit(1); } } while (0)

__global__ void copy16(const uint4 *__restrict__ src, uint4 *__restrict__ dst, long long nvec) {
    const long long nth = (long long)gridDim.x * blockDim.x;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * nth < nvec; i += 4 * nth) {
        const uint4 a = src[i], b = src[i + nth], c = src[i + 2 * nth], d = src[i + 3 * nth];
        dst[i] = a; dst[i + nth] = b; dst[i + 2 * nth] = c; dst[i + 3 * nth] = d;
    }
    for (; i < nvec; i += nth) dst[i] = src[i];
}

int main() {
    const size_t bytes = 1ull << 30;
    void *h_src, *h_dst, *d_a, *d_b;
    CK(cudaHostAlloc(&h_src, bytes, cudaHostAllocDefault));
    CK(cudaHostAlloc(&h_dst, bytes, cudaHostAllocDefault));
    CK(cudaMalloc(&d_a, bytes));
    CK(cudaMalloc(&d_b, bytes));
    for (size_t i = 0; i < bytes / 8; i += 4096) reinterpret_cast<uint64_t *>(h_src)[i] = i;
    CK(cudaMemset(d_a, 1, bytes));
    void *hs_dev, *hd_dev;   // device views of the pinned buffers
    CK(cudaHostGetDevicePointer(&hs_dev, h_src, 0));
    CK(cudaHostGetDevicePointer(&hd_dev, h_dst, 0));
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    cudaStream_t s1, s2;
    CK(cudaStreamCreate(&s1));
    CK(cudaStreamCreate(&s2));
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    auto timeit = [&](const char *name, double moved, auto launch) {
        launch();
        CK(cudaDeviceSynchronize());
        float best = 1e9f;
        for (int r = 0; r < 5; ++r) {
            CK(cudaEventRecord(e0, s1));
            launch();
            CK(cudaEventRecord(e1, s1));
            CK(cudaEventSynchronize(e1));
            CK(cudaDeviceSynchronize());
            float ms;
            CK(cudaEventElapsedTime(&ms, e0, e1));
            best = ms < best ? ms : best;
        }
        printf("%-58s %8.3f ms  %7.1f GB/s (bytes moved over the link)\n", name, best, moved / (best * 1e-3) / 1e9);
    };
    const long long nvec = (long long)(bytes / 16);
    timeit("memcpy H2D", bytes, [&] { CK(cudaMemcpyAsync(d_a, h_src, bytes, cudaMemcpyHostToDevice, s1)); });
    timeit("memcpy D2H", bytes, [&] { CK(cudaMemcpyAsync(h_dst, d_a, bytes, cudaMemcpyDeviceToHost, s1)); });
    timeit("memcpy H2D + D2H on two streams", 2.0 * bytes, [&] {
        CK(cudaMemcpyAsync(d_a, h_src, bytes, cudaMemcpyHostToDevice, s1));
        CK(cudaMemcpyAsync(h_dst, d_b, bytes, cudaMemcpyDeviceToHost, s2));
        cudaEvent_t j;
        CK(cudaEventCreateWithFlags(&j, cudaEventDisableTiming));
        CK(cudaEventRecord(j, s2));
        CK(cudaStreamWaitEvent(s1, j, 0));
        CK(cudaEventDestroy(j));
    });
    for (int per_sm : {2, 4}) {
        char nm[96];
        snprintf(nm, sizeof nm, "kernel reads host, writes device (%d CTAs/SM)", per_sm);
        timeit(nm, bytes, [&] { copy16<<<sms * per_sm, 512, 0, s1>>>((const uint4 *)hs_dev, (uint4 *)d_b, nvec); CK(cudaGetLastError()); });
        snprintf(nm, sizeof nm, "kernel reads device, writes host (%d CTAs/SM)", per_sm);
        timeit(nm, bytes, [&] { copy16<<<sms * per_sm, 512, 0, s1>>>((const uint4 *)d_a, (uint4 *)hd_dev, nvec); CK(cudaGetLastError()); });
        snprintf(nm, sizeof nm, "kernel reads host, writes host (%d CTAs/SM)", per_sm);
        timeit(nm, 2.0 * bytes, [&] { copy16<<<sms * per_sm, 512, 0, s1>>>((const uint4 *)hs_dev, (uint4 *)hd_dev, nvec); CK(cudaGetLastError()); });
    }
    return 0;
}
