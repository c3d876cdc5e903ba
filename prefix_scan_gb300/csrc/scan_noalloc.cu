// scan_noalloc.cu -- an int32 inclusive scan for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a device workspace: code that runs
// where cudaMalloc is forbidden or unavailable (inside a custom allocator
// or a memory-pool callback, in a plug-in whose host application owns all
// device memory, in a hot path that must never touch the allocator), or a
// caller that simply cannot size and keep a workspace buffer.  For them this
// file keeps the look-back scratch (the 256-byte header plus one status
// descriptor slot per tile) in a fixed array in the library's own device
// memory, so the call needs only the input and output.
//
// Consequences of a file-scope device array:
//   - every GPU that loads this library holds the array
//     (PS_NOALLOC_SCRATCH_BYTES, 4.5 MiB + 256 bytes) until the process exits;
//   - all calls on a device share it: two calls whose work overlaps on the
//     GPU (different streams, or different host threads without ordering)
//     race on it and give wrong results; calls on one stream are ordered and
//     safe;
//   - it keeps what the last call left there, which is exactly the state the
//     next call needs (a workspace is zero-filled once and every call leaves
//     it ready for the next); the first call on a device zero-fills it.
#include <cuda_runtime.h>

#include <mutex>

#include "prefix_scan.h"
#include "scan_internal.h"

namespace {

// The regular workspace size for the largest accepted n, so that the two
// can never drift apart; the header states the same number.
constexpr size_t kNoallocScratchBytes = ps::workspace_bytes(PS_INT32, (size_t)PS_NOALLOC_MAX_ELEMENTS);
static_assert(kNoallocScratchBytes <= (size_t)PS_NOALLOC_SCRATCH_BYTES,
              "the tile geometry changed: update PS_NOALLOC_SCRATCH_BYTES");

// The scratch itself.  Host code must not pass this name to a kernel: on
// the host it is only a stand-in symbol, not a device address.  The device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the device address of
// the scratch array and zero-fill it on the caller's stream.  Looking up the
// symbol may load the library's device code onto the device, which is why
// the first call on a device should not be made while a stream is being
// captured.
cudaError_t scratch_for_current_device(cudaStream_t stream, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        // a workspace starts zero-filled; device globals are, but make sure
        e = cudaMemsetAsync(p, 0, PS_NOALLOC_SCRATCH_BYTES, stream);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ps_status ps_scan_inclusive_i32_noalloc(const int32_t *in, int32_t *out, size_t n,
                                                   ps_stream_t stream) {
    if (n == 0) return PS_OK;
    if (n > (size_t)PS_NOALLOC_MAX_ELEMENTS) return PS_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const cudaError_t e = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (e != cudaSuccess) {
        ps::note_cuda_error(e);  // readable with ps_last_cuda_error()
        return PS_ERR_CUDA;
    }
    return ps_scan_inclusive_i32(in, out, n, scratch, PS_NOALLOC_SCRATCH_BYTES, stream);
}
