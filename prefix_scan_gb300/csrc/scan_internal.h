// scan_internal.h -- host-side pieces shared by the library's translation
// units: workspace layout, tile geometry, launcher declarations.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "prefix_scan.h"

namespace ps {

// ---- workspace layout ------------------------------------------------------
// [0, 256)                 header
// [256, 256 + D)           descriptor slots, one per tile of a single-pass scan
// [256 + D, 256 + D + P)   tile aggregates of the reduce-then-scan comparison
//                          path (its own region: it never disturbs descriptors)
//
// No call resets the workspace before it starts.  A workspace is zero-filled
// once, before its first use; from then on every call leaves it ready for the
// next: descriptors carry the number ("epoch") of the call that wrote them,
// so those of earlier calls read as "nothing published", and the last CTA of
// a call puts the tile counter back to 0 and advances the epoch.
struct Header {
    unsigned long long tile_counter;  // dynamic tile ids; 0 between calls
    unsigned long long status;        // epoch << 8 | ps_status of a device-side error
    unsigned long long capacity;      // largest ws_bytes any call declared (cleared on wrap)
    unsigned int done;                // CTAs finished in the running call; 0 between calls
    unsigned int epoch;               // number of this call, modulo 2^30
    unsigned int magic;               // 0 in a fresh workspace, kWorkspaceMagic once used
};
constexpr size_t kHeaderBytes = 256;
static_assert(sizeof(Header) <= kHeaderBytes, "header too large");
constexpr uint32_t kEpochBits = 30;
constexpr uint32_t kEpochMask = (1u << kEpochBits) - 1;
constexpr uint32_t kWorkspaceMagic = 0x50534742u;

// Tile geometry: THREADS scanning threads per tile, ITEMS elements per
// thread (in rows of 16-byte vectors): 8192-element tiles for 32-bit types,
// 4096 for int64 -- 32 KiB either way.  The look-back window is 32 lanes x
// LOOKBACK_K descriptors.  The persistent kernel keeps STAGES tiles of
// shared memory per CTA and runs CTAS_PER_SM CTAs per SM.  The macros only
// exist so that a tuning sweep can rebuild with other values.
#ifndef PS_THREADS
#define PS_THREADS 256
#endif
#ifndef PS_ITEMS32
#define PS_ITEMS32 32
#endif
#ifndef PS_ITEMS64
#define PS_ITEMS64 16
#endif
#ifndef PS_PERSIST_STAGES
#define PS_PERSIST_STAGES 3
#endif
#ifndef PS_PERSIST_CTAS_PER_SM
#define PS_PERSIST_CTAS_PER_SM 2
#endif
#ifndef PS_LOOKBACK_K
#define PS_LOOKBACK_K 1
#endif
// Poll back-off of the look-back: spin PS_SPIN_POLLS polls, then sleep
// PS_SLEEP_NS_SHORT per poll, and PS_SLEEP_NS_LONG once past
// PS_SLEEP_AFTER_LONG polls.  Sleeping keeps hundreds of spinning warps from
// saturating the L2 slices that hold neighbouring descriptors.
#ifndef PS_SPIN_POLLS
#define PS_SPIN_POLLS 8
#endif
#ifndef PS_SLEEP_NS_SHORT
#define PS_SLEEP_NS_SHORT 32
#endif
#ifndef PS_SLEEP_AFTER_LONG
#define PS_SLEEP_AFTER_LONG 64
#endif
#ifndef PS_SLEEP_NS_LONG
#define PS_SLEEP_NS_LONG 512
#endif
// Bytes between consecutive tile descriptors.  Packed 8-byte descriptors
// put 16 neighbouring tiles on one 128-byte L2 line, which every publish
// and every look-back of those tiles then contends for; spreading them to
// one per 64 bytes measured fastest over int32 and int64 on GB300.  64-bit
// types use at least 16.
#ifndef PS_DESC_STRIDE
#define PS_DESC_STRIDE 64
#endif
constexpr int kDescStride32 = PS_DESC_STRIDE;
constexpr int kDescStride64 = PS_DESC_STRIDE < 16 ? 16 : PS_DESC_STRIDE;
static_assert(PS_DESC_STRIDE % 8 == 0, "descriptor stride must be a multiple of 8");
constexpr int kThreads = PS_THREADS;
constexpr int kItems32 = PS_ITEMS32;   // int32 / fp32 elements per thread
constexpr int kItems64 = PS_ITEMS64;   // int64 elements per thread
constexpr int kLookbackK = PS_LOOKBACK_K;
constexpr int kPStages = PS_PERSIST_STAGES;
constexpr int kPCtasPerSm = PS_PERSIST_CTAS_PER_SM;

constexpr size_t tile_elems(ps_dtype dt) {
    return (size_t)kThreads * (dt == PS_INT64 ? kItems64 : kItems32);
}
constexpr size_t elem_bytes(ps_dtype dt) { return dt == PS_INT64 ? 8 : 4; }
constexpr size_t desc_bytes(ps_dtype dt) { return dt == PS_INT64 ? kDescStride64 : kDescStride32; }
constexpr size_t num_tiles(ps_dtype dt, size_t n) { return (n + tile_elems(dt) - 1) / tile_elems(dt); }
constexpr size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
constexpr size_t desc_region_bytes(ps_dtype dt, size_t n) {
    return round_up(num_tiles(dt, n) * desc_bytes(dt), 256);
}
constexpr size_t partials_offset(ps_dtype dt, size_t n) { return kHeaderBytes + desc_region_bytes(dt, n); }
constexpr size_t workspace_bytes(ps_dtype dt, size_t n) {
    if (n == 0) return 0;
    return partials_offset(dt, n) + round_up(num_tiles(dt, n) * 8, 256);
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

// Operator of a single-pass scan: the public ps_op values, and the two
// operators of the 8-byte pair element types (int64_t storage only).
enum ScanOpCode : int {
    kOpSum = PS_OP_SUM,
    kOpMax = PS_OP_MAX,
    kOpMin = PS_OP_MIN,
    kOpPairI32F32 = 16,   // {int32, fp32} pairs, field-wise sum
    kOpAffineF32 = 17     // fp32 affine maps {a, b}, composition
};

// Launch arguments common to the single-pass kernels.
struct PassArgs {
    const void *in;
    void *out;
    unsigned long long n;
    unsigned char *ws;             // workspace base (header + descriptors)
    const void *carry_in;          // optional device scalar added to every output
    void *carry_out;               // optional device scalar: inclusive total
    unsigned long long ws_bytes;   // workspace capacity (cleared when the epoch wraps)
    uint32_t max_polls;
};

// Enqueue the persistent TMA-fed single-pass kernel (16-byte aligned in/out).
template <typename T>
cudaError_t launch_persistent(const PassArgs &a, bool exclusive, int op, cudaStream_t s);

// Enqueue one single-pass scan (one kernel; the workspace needs no reset).
// T is int32_t, int64_t or float.  Decoupled look-back on 16-byte aligned
// arrays runs the persistent kernel; otherwise one CTA per tile.
template <typename T>
cudaError_t launch_single_pass(const PassArgs &a, bool exclusive, Lookback lb, cudaStream_t s,
                               int op = kOpSum);

// Short arrays (n <= small_scan_limit<T>(): two tiles) are scanned by one
// CTA with no look-back and no workspace update (csrc/scan_small.cu).
template <typename T>
unsigned long long small_scan_limit();
template <typename T>
cudaError_t launch_small(const PassArgs &a, bool exclusive, int op, cudaStream_t s);

// Third kernel of reduce-then-scan: tile scan seeded from the workspace.
template <typename T>
cudaError_t launch_seeded_tile_scan(const PassArgs &a, bool exclusive, cudaStream_t s);

// Enqueue the three-kernel reduce-then-scan comparison path.
template <typename T>
cudaError_t launch_reduce_then_scan(const void *in, void *out, unsigned long long n,
                                    unsigned char *ws, bool exclusive, cudaStream_t s);

// Test hook: run the look-back alone for `tile` over a prepared descriptor
// array (one warp) as call `epoch`, writing the exclusive prefix and a
// status word.
template <typename T>
cudaError_t launch_lookback_probe(const void *desc, long long tile, uint32_t epoch,
                                  uint32_t max_polls, void *result, unsigned long long *status,
                                  cudaStream_t s);

// Launch arguments of the compaction kernels (select / partition).
struct SelectArgs {
    const void *in;
    const uint8_t *flags;
    void *out;
    unsigned long long n;
    unsigned char *ws;
    unsigned long long ws_bytes;
    unsigned long long *num_selected;   // device, may be null
    unsigned long long threshold_bits;  // the threshold's bits (greater / less)
    uint32_t max_polls;
    int use_bulk;                       // values (and flags) 16-byte aligned
};

// Enqueue a single-pass select or partition; op: 0 flag array, 1 nonzero,
// 2 greater than the threshold, 3 less than the threshold.
template <typename T>
cudaError_t launch_select(const SelectArgs &a, int op, bool partition, cudaStream_t s);

// Reduce-by-key / run-length encoding: tiles of 4096 elements for 32-bit
// keys, 2048 for 64-bit keys (16 KiB of keys plus their 32-bit values per
// tile), one 16-byte two-word descriptor slot per tile holding the (run
// count, run value) pair.
constexpr size_t rbk_tile_elems(ps_dtype key_dt) { return key_dt == PS_INT64 ? 2048 : 4096; }
constexpr size_t rbk_num_tiles(ps_dtype key_dt, size_t n) {
    return (n + rbk_tile_elems(key_dt) - 1) / rbk_tile_elems(key_dt);
}
constexpr size_t rbk_workspace_bytes(ps_dtype key_dt, size_t n) {
    if (n == 0) return 0;
    return kHeaderBytes + round_up(rbk_num_tiles(key_dt, n) * kDescStride64, 256);
}

struct RbkArgs {
    const void *keys;
    const void *vals;                   // null: run-length encoding (every value is 1)
    void *unique_keys;
    void *aggs;
    unsigned long long n;
    unsigned char *ws;
    unsigned long long ws_bytes;
    unsigned long long *num_runs;       // device, may be null
    uint32_t max_polls;
    int use_bulk;                       // keys and values 16-byte aligned
};

// Enqueue a single-pass reduce-by-key (vals != null) or run-length encoding.
// key_dt: PS_INT32 / PS_FLOAT32 (32-bit keys) or PS_INT64; val_dt: PS_INT32
// or PS_FLOAT32.
cudaError_t launch_reduce_by_key(const RbkArgs &a, ps_dtype key_dt, ps_dtype val_dt, cudaStream_t s);

// Enqueue a single-pass run-length encoding (a.vals unused): tiles of 32 KiB
// of keys, so the reduce-by-key workspace size covers it.
cudaError_t launch_run_length_encode(const RbkArgs &a, ps_dtype key_dt, cudaStream_t s);

// Trace build (PS_TRACE): each kernel's translation unit copies the trace of
// its own last launch (cudaErrorNotSupported in the product build).
cudaError_t trace_copy_scan(uint64_t *ts, uint32_t *lookback, int32_t *cta, size_t tiles);
cudaError_t trace_copy_scan_ctas(uint64_t *ts, size_t ctas);
cudaError_t trace_copy_select(uint64_t *ts, uint32_t *lookback, int32_t *cta, size_t tiles);
cudaError_t trace_copy_select_ctas(uint64_t *ts, size_t ctas);
cudaError_t trace_copy_rbk(uint64_t *ts, uint32_t *lookback, int32_t *cta, size_t tiles);
cudaError_t trace_copy_rbk_ctas(uint64_t *ts, size_t ctas);
cudaError_t trace_copy_rle(uint64_t *ts, uint32_t *lookback, int32_t *cta, size_t tiles);
cudaError_t trace_copy_rle_ctas(uint64_t *ts, size_t ctas);

// Records `e` as the calling thread's last CUDA error (ps_last_cuda_error).
void note_cuda_error(cudaError_t e);

// The checked body of ps_scan_seeded (decoupled look-back with carries).
ps_status scan_seeded(ps_dtype dt, int exclusive, const void *in, void *out, size_t n,
                      const void *carry_in, void *carry_out, void *ws, size_t ws_bytes,
                      cudaStream_t s);

}  // namespace ps
