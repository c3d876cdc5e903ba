// scan_host.cu -- scan of arrays in HOST memory, streamed through the GPU.
//
// The array is cut into chunks of 32 MiB.  Each chunk is copied to one of
// three device staging buffers, scanned there in place with the seeded
// single-pass scan (the carry -- the running total of all earlier chunks --
// lives in device memory after the staging buffers, so no chunk waits for
// the host), and copied back.  Three streams overlap the host-to-device
// copy of chunk i+1, the scan of chunk i and the device-to-host copy of
// chunk i-1, so the two directions of the host link run at the same time.
// The caller's stream runs the scans and, at the end, waits for the last
// copy, so work after this call on that stream sees the whole result.
#include <cuda_runtime.h>

#include <cstdint>

#include "prefix_scan.h"
#include "scan_internal.h"

namespace {

// Chunk size: the first chunk's host-to-device copy and the last chunk's
// device-to-host copy run alone, so smaller chunks shorten the pipeline's
// fill and drain; each chunk costs one scan launch.  (A macro so that a
// tuning sweep can rebuild with other sizes.)
#ifndef PS_HOST_CHUNK_MIB
#define PS_HOST_CHUNK_MIB 32
#endif
constexpr size_t kChunkBytes = (size_t)PS_HOST_CHUNK_MIB << 20;
// Device staging buffers the chunks rotate through: with more than two,
// host-to-device copies can run ahead while a chunk is scanned.
#ifndef PS_HOST_BUFFERS
#define PS_HOST_BUFFERS 3
#endif
constexpr int kBuffers = PS_HOST_BUFFERS;
static_assert(kBuffers >= 2 && kBuffers <= 8, "2 to 8 staging buffers");

bool host_dtype_ok(int dt) { return dt == PS_INT32 || dt == PS_INT64 || dt == PS_FLOAT32; }
size_t chunk_elems(ps_dtype dt) { return kChunkBytes / ps::elem_bytes(dt); }
size_t stage_bytes(ps_dtype dt, size_t n) {
    const size_t c = n < chunk_elems(dt) ? n : chunk_elems(dt);
    return ps::round_up(c * ps::elem_bytes(dt), 256);
}

struct Pipeline {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[kBuffers] = {}, scanned[kBuffers] = {}, freed[kBuffers] = {};

    cudaError_t create() {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t *ev : {&start, &done})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int b = 0; b < kBuffers; ++b)
            for (cudaEvent_t *ev : {&loaded[b], &scanned[b], &freed[b]})
                if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
        return cudaSuccess;
    }
    // Resources are released once their pending work completes.
    ~Pipeline() {
        for (cudaEvent_t ev : {start, done})
            if (ev) cudaEventDestroy(ev);
        for (int b = 0; b < kBuffers; ++b)
            for (cudaEvent_t ev : {loaded[b], scanned[b], freed[b]})
                if (ev) cudaEventDestroy(ev);
        if (h2d) cudaStreamDestroy(h2d);
        if (d2h) cudaStreamDestroy(d2h);
    }
};

}  // namespace

extern "C" size_t ps_scan_host_staging_size(ps_dtype dtype, size_t n) {
    if (!host_dtype_ok(dtype) || n == 0) return 0;
    return kBuffers * stage_bytes(dtype, n) + 256;
}

extern "C" ps_status ps_scan_host(ps_dtype dtype, int exclusive, const void *h_in, void *h_out,
                                  size_t n, void *d_staging, size_t staging_bytes, void *ws,
                                  size_t ws_bytes, ps_stream_t stream) {
    if (!host_dtype_ok(dtype)) return PS_ERR_INVALID_ARG;
    if (n == 0) return PS_OK;
    if (h_in == nullptr || h_out == nullptr || d_staging == nullptr || ws == nullptr)
        return PS_ERR_INVALID_ARG;
    const size_t es = ps::elem_bytes(dtype);
    if ((reinterpret_cast<uintptr_t>(h_in) | reinterpret_cast<uintptr_t>(h_out)) % es != 0 ||
        reinterpret_cast<uintptr_t>(d_staging) % 256 != 0)
        return PS_ERR_INVALID_ARG;
    if (n > (SIZE_MAX / 2) / es) return PS_ERR_INVALID_ARG;
    const size_t bytes = n * es;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(h_in), b0 = reinterpret_cast<uintptr_t>(h_out);
    if (h_in != h_out && a0 < b0 + bytes && b0 < a0 + bytes) return PS_ERR_OVERLAP;
    if (staging_bytes < ps_scan_host_staging_size(dtype, n)) return PS_ERR_WORKSPACE_TOO_SMALL;
    const size_t C = chunk_elems(dtype);
    if (ws_bytes < ps::workspace_bytes(dtype, n < C ? n : C)) return PS_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t s = (cudaStream_t)stream;
    unsigned char *stage[kBuffers];
    for (int b = 0; b < kBuffers; ++b) stage[b] = static_cast<unsigned char *>(d_staging) + b * stage_bytes(dtype, n);
    void *carry = static_cast<unsigned char *>(d_staging) + kBuffers * stage_bytes(dtype, n);
    const unsigned char *src = static_cast<const unsigned char *>(h_in);
    unsigned char *dst = static_cast<unsigned char *>(h_out);

    Pipeline p;
    cudaError_t e = p.create();
    ps_status st = PS_OK;
    // the copy streams start after the work already queued on the caller's stream
    if (e == cudaSuccess) e = cudaMemsetAsync(carry, 0, es, s);
    if (e == cudaSuccess) e = cudaEventRecord(p.start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.h2d, p.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.start, 0);
    const size_t chunks = (n + C - 1) / C;
    for (size_t i = 0; i < chunks && e == cudaSuccess && st == PS_OK; ++i) {
        const int b = (int)(i % kBuffers);
        const size_t off = i * C, len = (n - off < C) ? n - off : C;
        if (i >= (size_t)kBuffers) e = cudaStreamWaitEvent(p.h2d, p.freed[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(stage[b], src + off * es, len * es, cudaMemcpyHostToDevice, p.h2d);
        if (e == cudaSuccess) e = cudaEventRecord(p.loaded[b], p.h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p.loaded[b], 0);
        if (e != cudaSuccess) break;
        st = ps::scan_seeded(dtype, exclusive, stage[b], stage[b], len, carry, carry, ws, ws_bytes, s);
        if (st != PS_OK) break;
        e = cudaEventRecord(p.scanned[b], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.scanned[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst + off * es, stage[b], len * es, cudaMemcpyDeviceToHost, p.d2h);
        if (e == cudaSuccess) e = cudaEventRecord(p.freed[b], p.d2h);
    }
    // join: the caller's stream waits for everything enqueued above
    cudaError_t e2 = cudaEventRecord(p.done, p.d2h);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, p.done, 0);
    cudaError_t e3 = cudaEventRecord(p.done, p.h2d);
    if (e3 == cudaSuccess) e3 = cudaStreamWaitEvent(s, p.done, 0);
    if (st != PS_OK) return st;
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = e3;
    if (e != cudaSuccess) {
        ps::note_cuda_error(e);
        return PS_ERR_CUDA;
    }
    return PS_OK;
}
