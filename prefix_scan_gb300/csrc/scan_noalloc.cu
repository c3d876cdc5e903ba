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
//   - cudaDeviceReset destroys the device's context and with it the loaded
//     copy of the array; the next call finds a fresh (zeroed) copy, possibly
//     at another address, which is why every call looks the address up.
#include <cuda_runtime.h>

#include <mutex>

#include "prefix_scan.h"
#include "prefix_scan_testing.h"
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
void *g_scratch_ptr[kMaxDevices] = {};   // address the set-up zero-filled, per device

// With the device current: the device address of the scratch array.  The
// look-up runs on every call, because the address belongs to the device's
// current context: after cudaDeviceReset the library's device code is loaded
// again and the array may sit elsewhere.  Set-up, once per device and again
// whenever the address moved: zero-fill the array on the caller's stream.
// The first look-up on a device may load the library's device code onto it,
// which is why the first call on a device should not be made while a
// stream is being captured.
cudaError_t scratch_for_current_device(cudaStream_t stream, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] != p) {
        // a workspace starts zero-filled; a freshly loaded device array is,
        // but make sure
        e = cudaMemsetAsync(p, 0, PS_NOALLOC_SCRATCH_BYTES, stream);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = p;
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

// Test hook: the device address of the current device's scratch array, so
// that a test can read its status word with ps_get_device_status.
extern "C" ps_status ps_testing_noalloc_scratch(void **scratch, ps_stream_t stream) {
    if (scratch == nullptr) return PS_ERR_INVALID_ARG;
    const cudaError_t e = scratch_for_current_device((cudaStream_t)stream, scratch);
    if (e != cudaSuccess) {
        ps::note_cuda_error(e);
        return PS_ERR_CUDA;
    }
    return PS_OK;
}
