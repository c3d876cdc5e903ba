// scan_internal.h -- host-side pieces shared by the library's translation
// units: workspace layout, tile geometry, launcher declarations.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "prefix_scan.h"

namespace ps {

// ---- workspace layout ------------------------------------------------------
// [0, 256)        header: tile counter, status word, carry slots
// [256, ...)      one status descriptor per tile (8 B for 32-bit types,
//                 16 B for 64-bit types), or the tile aggregates of the
//                 reduce-then-scan comparison path (same footprint).
struct Header {
    unsigned long long tile_counter;  // dynamic tile ids (atomicAdd)
    unsigned int status;              // ps_status written by the device
    unsigned int pad0;
    unsigned long long carry[4];      // device-side carries (host streaming)
};
constexpr size_t kHeaderBytes = 256;
static_assert(sizeof(Header) <= kHeaderBytes, "header too large");

// Tile geometry of the decoupled look-back path: THREADS threads per CTA,
// ITEMS consecutive-in-rows elements per thread.
constexpr int kThreads = 256;
constexpr int kItems32 = 16;   // int32 / fp32: 4096-element tiles (16 KiB)
constexpr int kItems64 = 8;    // int64: 2048-element tiles (16 KiB)

inline size_t tile_elems(ps_dtype dt) {
    return (size_t)kThreads * (dt == PS_INT64 ? kItems64 : kItems32);
}
inline size_t elem_bytes(ps_dtype dt) { return dt == PS_INT64 ? 8 : 4; }
inline size_t desc_bytes(ps_dtype dt) { return dt == PS_INT64 ? 16 : 8; }
inline size_t num_tiles(ps_dtype dt, size_t n) { return (n + tile_elems(dt) - 1) / tile_elems(dt); }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline size_t workspace_bytes(ps_dtype dt, size_t n) {
    if (n == 0) return 0;
    return kHeaderBytes + round_up(num_tiles(dt, n) * desc_bytes(dt), 256);
}

// Default cap on look-back polls before a CTA gives up (each poll is at
// least one L2 round trip; with the back-off this bounds a wait to seconds).
constexpr uint32_t kDefaultMaxPolls = 1u << 21;

// Where a tile's exclusive prefix comes from in the tile-scan kernel:
//   Decoupled   warp-parallel decoupled look-back (the product path);
//   Chained     wait for the immediate predecessor's inclusive prefix;
//   Precomputed read it from the workspace (third kernel of the
//               reduce-then-scan comparison path; tile id = blockIdx.x).
enum class Lookback { Decoupled = 0, Chained = 1, Precomputed = 2 };

// Launch arguments common to the single-pass kernels.
struct PassArgs {
    const void *in;
    void *out;
    unsigned long long n;
    unsigned char *ws;             // workspace base (header + descriptors)
    const void *carry_in;          // optional device scalar added to every output
    void *carry_out;               // optional device scalar: inclusive total
    uint32_t max_polls;
};

// Enqueue one single-pass scan (workspace reset + kernel).  T is int32_t,
// int64_t or float.
template <typename T>
cudaError_t launch_single_pass(const PassArgs &a, bool exclusive, Lookback lb, cudaStream_t s);

// Third kernel of reduce-then-scan: tile scan seeded from the workspace.
template <typename T>
cudaError_t launch_seeded_tile_scan(const PassArgs &a, bool exclusive, cudaStream_t s);

// Enqueue the three-kernel reduce-then-scan comparison path.
template <typename T>
cudaError_t launch_reduce_then_scan(const void *in, void *out, unsigned long long n,
                                    unsigned char *ws, bool exclusive, cudaStream_t s);

// Test hook: run the look-back alone for `tile` over a prepared descriptor
// array (one warp), writing the exclusive prefix and a status word.
template <typename T>
cudaError_t launch_lookback_probe(const void *desc, long long tile, uint32_t max_polls,
                                  void *result, unsigned int *status, cudaStream_t s);

// Records `e` as the calling thread's last CUDA error (ps_last_cuda_error).
void note_cuda_error(cudaError_t e);

}  // namespace ps
