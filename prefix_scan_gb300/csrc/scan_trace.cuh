// scan_trace.cuh -- the pipeline trace of the persistent kernels (trace
// build only).
//
// Built with PS_TRACE defined, a kernel records for each of the first
// PS_TRACE_TILES tiles of its launch the %globaltimer at eight hand-offs of
// its pipeline (claim, data landed, A published, look-back start, P
// published, compute start, prefix received, stores issued), the CTA that
// took it, and the look-back's windows and re-polls; per CTA its start,
// header verdict and end.  One store per point by one lane.  Every
// translation unit that includes this header has buffers of its own
// (internal linkage), read back by the TRACE_COPY_FUNCTIONS it defines, so
// the scan, select, reduce-by-key and run-length kernels each keep the
// trace of their own last launch.  Without PS_TRACE none of it is compiled.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "prefix_scan_trace.h"
#include "scan_pipeline.cuh"

namespace ps {

#ifdef PS_TRACE
namespace {
constexpr long long kTraceTiles = PS_TRACE_TILES;
constexpr int kTraceCtas = PS_TRACE_CTAS;
__device__ unsigned long long g_trace_ts[kTraceTiles][PS_TRACE_POINTS];
__device__ uint32_t g_trace_lookback[kTraceTiles];
__device__ int g_trace_cta[kTraceTiles];
__device__ unsigned long long g_trace_cta_ts[kTraceCtas][PS_TRACE_CTA_POINTS];

__device__ __forceinline__ void trace_cta_point(int k) {
    if (blockIdx.x < kTraceCtas) g_trace_cta_ts[blockIdx.x][k] = global_ns();
}
__device__ __forceinline__ void trace_point(long long tile, int k) {
    if (tile >= 0 && tile < kTraceTiles) g_trace_ts[tile][k] = global_ns();
}
__device__ __forceinline__ uint32_t *trace_lookback_slot(long long tile) {
    return (tile >= 0 && tile < kTraceTiles) ? &g_trace_lookback[tile] : nullptr;
}
__device__ __forceinline__ void trace_cta(long long tile) {
    if (tile >= 0 && tile < kTraceTiles) g_trace_cta[tile] = (int)blockIdx.x;
}

// Host side: copies of this translation unit's buffers (after a device
// synchronisation).
__attribute__((unused)) cudaError_t trace_copy_tiles(uint64_t *ts, uint32_t *lookback, int32_t *cta,
                                                     size_t tiles) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(ts, g_trace_ts, tiles * sizeof(g_trace_ts[0]));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(lookback, g_trace_lookback, tiles * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(cta, g_trace_cta, tiles * sizeof(int32_t));
    return e;
}
__attribute__((unused)) cudaError_t trace_copy_ctas(uint64_t *ts, size_t ctas) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(ts, g_trace_cta_ts, ctas * sizeof(g_trace_cta_ts[0]));
    return e;
}
}  // namespace
#define PS_TRACE_POINT(tile, k) trace_point((tile), (k))
#define PS_TRACE_CTA(tile) trace_cta(tile)
#define PS_TRACE_LOOKBACK(tile) trace_lookback_slot(tile)
#define PS_TRACE_CTA_POINT(k) trace_cta_point(k)
// Defines the translation unit's two read-back functions under the given
// names (declared in scan_internal.h).
#define TRACE_COPY_FUNCTIONS(tiles_fn, ctas_fn)                                                   \
    cudaError_t tiles_fn(uint64_t *ts, uint32_t *lb, int32_t *cta, size_t tiles) {              \
        return trace_copy_tiles(ts, lb, cta, tiles);                                            \
    }                                                                                           \
    cudaError_t ctas_fn(uint64_t *ts, size_t ctas) { return trace_copy_ctas(ts, ctas); }
#else
#define PS_TRACE_POINT(tile, k) ((void)0)
#define PS_TRACE_CTA(tile) ((void)0)
#define PS_TRACE_LOOKBACK(tile) nullptr
#define PS_TRACE_CTA_POINT(k) ((void)0)
#define TRACE_COPY_FUNCTIONS(tiles_fn, ctas_fn)                                                   \
    cudaError_t tiles_fn(uint64_t *, uint32_t *, int32_t *, size_t) { return cudaErrorNotSupported; } \
    cudaError_t ctas_fn(uint64_t *, size_t) { return cudaErrorNotSupported; }
#endif

}  // namespace ps
