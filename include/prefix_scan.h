/*
 * prefix_scan.h -- C ABI of the GB300 (sm_103a) device-wide prefix sum.
 *
 * The operation (problem statement of the RTX 4090 scan tutorial,
 * "smarter.xin/posts/bcb510f9", section 1; "Prefix Sum" definition of the
 * page "CUDA-Operators-6-Cumsum", section 1):
 *
 *     inclusive   y[i] = x[0] + x[1] + ... + x[i]          0 <= i < n
 *     exclusive   y[0] = 0,  y[i] = x[0] + ... + x[i-1]
 *                 (conversion section "Inclusive 与 Exclusive 的转换" of the
 *                  same tutorial)
 *
 * computed in ONE pass over the data by the single-pass scan with decoupled
 * look-back ("Single-pass Parallel Prefix Scan with Decoupled Look-back",
 * Merrill & Garland, summary page, sections 4.1 and 4.4): every input
 * element is read once and every output element written once (~2n words).
 *
 * Arithmetic:
 *   int32 / int64  two's-complement wraparound, i.e. the exact sum modulo
 *                  2^32 / 2^64; results are bit-exact and deterministic.
 *   fp32           IEEE single-precision additions.  The association order
 *                  depends on run-time scheduling (section A6 of the paper
 *                  summary), so results may differ in the last bits from run
 *                  to run; NaN and Inf propagate as in IEEE arithmetic.
 *
 * Conventions shared by every entry point:
 *   - All data pointers (in, out, ws) are DEVICE pointers owned by the
 *     caller; the library allocates no device memory and keeps no state
 *     between calls.
 *   - `in`/`out` are contiguous arrays of n elements, aligned to their
 *     element size.  16-byte aligned arrays take the vectorised path.
 *   - in == out is an in-place scan and is allowed.  Any other overlap of
 *     the two arrays, or of either with the workspace, is rejected with
 *     PS_ERR_OVERLAP before anything is enqueued.
 *   - `ws` is a scratch workspace of at least ps_scan_workspace_size(dtype,
 *     n) bytes, 16-byte aligned.  It must be ZERO-FILLED ONCE before its
 *     first use (ps_workspace_init, cudaMemset, or a zeroed allocation) and
 *     then left alone between calls: no call resets it, each call leaves it
 *     ready for the next (any dtype, algorithm or n it is large enough for).
 *     A workspace that was never zero-filled makes the kernels do nothing
 *     and ps_get_device_status report PS_ERR_WORKSPACE_NOT_INITIALIZED.
 *     After an error from a call or from ps_get_device_status, zero it
 *     again.  Two calls that may run at the same time must not share one.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting for it.
 *   - n == 0 returns PS_OK, touches nothing and accepts NULL pointers.
 *   - Errors detected on the host are returned before anything is
 *     enqueued.  A failed CUDA runtime call yields PS_ERR_CUDA; its
 *     cudaError_t is kept per thread and read with ps_last_cuda_error().
 *   - A look-back that waits too long for a predecessor (which a correct
 *     launch never does) gives up instead of hanging: the kernel records
 *     PS_ERR_LOOKBACK_TIMEOUT in the workspace, writes unspecified output
 *     and finishes.  Read it with ps_get_device_status().
 *   - One kernel launch per scan (three for reduce-then-scan): there is no
 *     per-call workspace reset, because each tile descriptor carries the
 *     number of the call that wrote it (see ps_workspace_init).  The device
 *     entry points never synchronise, so they can be captured in a CUDA
 *     graph and the graph replayed any number of times.
 */
#ifndef PREFIX_SCAN_H
#define PREFIX_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA
 * headers. */
struct CUstream_st;
typedef struct CUstream_st *ps_stream_t;

typedef enum ps_status {
    PS_OK = 0,
    PS_ERR_INVALID_ARG = 1,         /* NULL pointer with n > 0, bad enum, misaligned pointer */
    PS_ERR_WORKSPACE_TOO_SMALL = 2, /* ws_bytes < ps_scan_workspace_size(dtype, n) */
    PS_ERR_OVERLAP = 3,             /* partial overlap of in/out, or ws overlapping either */
    PS_ERR_CUDA = 4,                /* a CUDA runtime call failed: see ps_last_cuda_error() */
    PS_ERR_LOOKBACK_TIMEOUT = 5,    /* device side: a look-back gave up waiting */
    PS_ERR_WORKSPACE_NOT_INITIALIZED = 6 /* device side: workspace never zero-filled */
} ps_status;

typedef enum ps_dtype { PS_INT32 = 0, PS_INT64 = 1, PS_FLOAT32 = 2 } ps_dtype;

/*
 * Bytes of workspace a scan of n elements of `dtype` needs (0 for n == 0):
 * a 256-byte header (tile counter, call number, status word) plus one
 * 64-byte slot per tile holding its status descriptor (section 4.1,
 * "partition descriptor": status flag X/A/P plus a value) and 8 bytes per
 * tile for the reduce-then-scan comparison path.  Tiles are 8192 elements
 * (32-bit types) or 4096 (int64), so about n/114 bytes (n/57 for int64).
 * The same size serves every algorithm below.
 */
size_t ps_scan_workspace_size(ps_dtype dtype, size_t n);

/*
 * Zero-fills `ws_bytes` bytes of workspace on `stream` (asynchronous): the
 * one preparation a workspace needs before its first scan, and after an
 * error.  Equivalent to cudaMemsetAsync(ws, 0, ws_bytes, stream).
 */
ps_status ps_workspace_init(void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Single-pass decoupled look-back scans (the product path).
 * in   : device array of n input elements (read once)
 * out  : device array of n output elements (written once; may equal in)
 * n    : number of elements (any value up to 2^62)
 * ws   : device workspace of ws_bytes >= ps_scan_workspace_size(...)
 * stream: CUDA stream the work is enqueued on
 */
ps_status ps_scan_inclusive_i32(const int32_t *in, int32_t *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_exclusive_i32(const int32_t *in, int32_t *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_inclusive_i64(const int64_t *in, int64_t *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_exclusive_i64(const int64_t *in, int64_t *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_inclusive_f32(const float *in, float *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_exclusive_f32(const float *in, float *out, size_t n,
                                void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Scans with other associative operators (section 4.2 of the paper
 * summary: the method combines only contiguous parts, in order):
 *   PS_OP_SUM  y[i] = x[0] + ... + x[i]        (the scans above)
 *   PS_OP_MAX  y[i] = max(x[0], ..., x[i])     exclusive y[0] = the lowest
 *   PS_OP_MIN  y[i] = min(x[0], ..., x[i])     value (INT_MIN, -inf) / the
 *                                              highest (INT_MAX, +inf)
 * Integers compare as signed.  fp32 max/min follow fmaxf/fminf: NaN
 * elements are skipped, so y[i] is the max/min of the non-NaN elements so
 * far (the identity if there is none); results are exact and identical
 * from run to run.  Decoupled look-back, same conventions, workspace and
 * errors as the scans above.
 */
typedef enum ps_op { PS_OP_SUM = 0, PS_OP_MAX = 1, PS_OP_MIN = 2 } ps_op;
ps_status ps_scan_op(ps_op op, ps_dtype dtype, int exclusive, const void *in, void *out, size_t n,
                     void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Global scan strategies.  PS_ALGO_DECOUPLED_LOOKBACK is the product path
 * (the six named entry points above).  The other two exist for comparison
 * only (paper summary, section 3.2 "global scan strategies"):
 *   PS_ALGO_REDUCE_THEN_SCAN  three kernels -- tile reductions, a scan of
 *                             the tile aggregates, a seeded re-scan of the
 *                             input -- about 3n words of traffic;
 *   PS_ALGO_CHAINED           single pass whose look-back waits for the
 *                             immediate predecessor's inclusive prefix only
 *                             (the "domino" scan with adjacent
 *                             synchronisation of the PMPP single-pass page).
 * PS_ALGO_REDUCE_THEN_SCAN is also the DETERMINISTIC mode: its additions
 * are associated in a fixed order (tile reductions, one CTA scanning the
 * tile aggregates, seeded tile scans), so fp32 results are bitwise
 * reproducible from run to run, which the single pass's look-back -- whose
 * order depends on scheduling -- does not give.  It costs about 3n words
 * of traffic instead of 2n.
 */
typedef enum ps_algo {
    PS_ALGO_DECOUPLED_LOOKBACK = 0,
    PS_ALGO_REDUCE_THEN_SCAN = 1,
    PS_ALGO_CHAINED = 2
} ps_algo;

/*
 * Generic form of the scans above: `exclusive` selects the scan kind
 * (0 = inclusive), in/out point to n elements of `dtype`.  Same
 * conventions and errors; PS_ERR_INVALID_ARG for an unknown algo/dtype.
 */
ps_status ps_scan(ps_algo algo, ps_dtype dtype, int exclusive, const void *in, void *out,
                  size_t n, void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Seeded scan: the decoupled look-back scan of `in` with a carry added to
 * every output, and the running total written back.  It is what a scan of
 * an array cut into pieces needs (a stream of chunks, shards on several
 * GPUs): piece i is scanned with the total of pieces 0..i-1 as its carry.
 *   carry_in  : device pointer to one element of `dtype` added to every
 *               output (exclusive: y[0] = *carry_in); NULL means 0.
 *   carry_out : device pointer receiving *carry_in + x[0] + ... + x[n-1];
 *               NULL means not written.  May equal carry_in.
 * Same conventions and errors as ps_scan; PS_ERR_OVERLAP if a carry lies
 * inside in, out or ws.  n == 0 copies *carry_in (or 0) to *carry_out.
 */
ps_status ps_scan_seeded(ps_dtype dtype, int exclusive, const void *in, void *out, size_t n,
                         const void *carry_in, void *carry_out, void *ws, size_t ws_bytes,
                         ps_stream_t stream);

/*
 * Scan of arrays in HOST memory (the end-to-end path).  The array is
 * streamed through the GPU in 32 MiB chunks rotating through three device
 * buffers: host-to-device copies of the next chunks, the seeded scan of
 * chunk i and the device-to-host copy of an earlier chunk run at the same
 * time on three streams, and the running total is carried on the device
 * from chunk to chunk.
 *   h_in, h_out : host arrays of n elements (h_out == h_in scans in place);
 *                 page-locked memory lets the copies overlap, pageable
 *                 memory works but the copies then serialise.
 *   d_staging   : device buffer of at least ps_scan_host_staging_size(dtype,
 *                 n) bytes, 256-byte aligned (three chunk buffers of up to
 *                 32 MiB + a carry).
 *   ws          : device workspace of at least ps_scan_workspace_size(dtype,
 *                 min(n, chunk)) bytes; ps_scan_workspace_size(dtype, n)
 *                 always suffices.
 * Work is enqueued on `stream`; the call returns before it completes and
 * h_out is complete once `stream` has reached this point (e.g. after
 * cudaStreamSynchronize).  Internal streams and events are created and
 * released by the call.  h_in and h_out must not change until then.
 */
size_t ps_scan_host_staging_size(ps_dtype dtype, size_t n);
ps_status ps_scan_host(ps_dtype dtype, int exclusive, const void *h_in, void *h_out, size_t n,
                       void *d_staging, size_t staging_bytes, void *ws, size_t ws_bytes,
                       ps_stream_t stream);

/*
 * Stream compaction in one pass (decoupled look-back paper summary,
 * section 4.4, "in-place compaction behaviour"): the output position of a
 * kept element is the exclusive prefix sum of the 0/1 keep flags, computed
 * by the same single-pass look-back and fused with the scatter.
 *   op         PS_SELECT_FLAGGED  keep x[i] where flags[i] != 0
 *              PS_SELECT_NONZERO  keep x[i] != 0
 *              PS_SELECT_GREATER  keep x[i] >  *threshold
 *              PS_SELECT_LESS     keep x[i] <  *threshold
 *              (fp32 compares per IEEE: NaN is never kept by GREATER/LESS,
 *              and is kept by NONZERO; -0.0 counts as zero)
 *   in         device array of n elements of `dtype`
 *   flags      device array of n bytes (PS_SELECT_FLAGGED only, else NULL)
 *   threshold  HOST pointer to one element of `dtype` (GREATER / LESS only)
 *   out        device array of n elements
 *   num_selected  device uint64 receiving the number kept (may be NULL)
 *   ws         workspace as for the scans: ps_scan_workspace_size(dtype, n)
 * ps_select writes the kept elements, in order, to out[0 .. count); the rest
 * of `out` is left untouched.  out == in compacts in place: safe in a single
 * pass because a tile learns its output offset only after every earlier
 * tile has loaded its input (needs in and flags 16-byte aligned, else
 * PS_ERR_OVERLAP).  ps_partition writes the kept elements to the front in
 * order and the others from the back in reverse order (the j-th rejected
 * element goes to out[n-1-j]), so `out` holds a permutation of `in`; out
 * must not overlap in.  n must be below 2^32.  Other conventions as for the
 * scans.
 */
typedef enum ps_select_op {
    PS_SELECT_FLAGGED = 0,
    PS_SELECT_NONZERO = 1,
    PS_SELECT_GREATER = 2,
    PS_SELECT_LESS = 3
} ps_select_op;
ps_status ps_select(ps_dtype dtype, ps_select_op op, const void *in, const uint8_t *flags,
                    const void *threshold, void *out, uint64_t *num_selected, size_t n, void *ws,
                    size_t ws_bytes, ps_stream_t stream);
ps_status ps_partition(ps_dtype dtype, ps_select_op op, const void *in, const uint8_t *flags,
                       const void *threshold, void *out, uint64_t *num_selected, size_t n,
                       void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Scans of 8-byte pair elements.  The decoupled look-back applies the
 * reduction operator only to contiguous inputs or partials (Merrill &
 * Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back",
 * section 4.2), so any associative operator works, commutative or not; the
 * paper's evaluation data include {int32, fp32} pairs (section A4).
 *
 * ps_scan_pair_i32_f32: field-wise sums, out[k] = {sum of in[0..k].i modulo
 * 2^32, sum of in[0..k].f in fp32 (association as in the fp32 scan)}.
 * ps_scan_affine_f32: each element is the map x -> a x + b; out[k] is the
 * composition of maps 0..k applied in order (map 0 first):
 *     out[k] = {a_k A_{k-1},  a_k B_{k-1} + b_k}  (fp32; identity {1, 0}),
 * so out[k].b is the k-th term of the recurrence y_k = a_k y_{k-1} + b_k
 * with y_{-1} = 0.  Exclusive: out[0] is the identity and out[k] the
 * composition of maps 0..k-1.
 *
 * Both are ps_scan_* with 8-byte elements: in and out 8-byte aligned
 * (16-byte alignment of both selects the bulk-copy kernel), out == in scans
 * in place, partial overlap is PS_ERR_OVERLAP, and the workspace is
 * ps_scan_workspace_size(PS_INT64, n) bytes with the same conventions.
 */
typedef struct ps_pair_i32_f32 {
    int32_t i;
    float f;
} ps_pair_i32_f32;
typedef struct ps_affine_f32 {
    float a;
    float b;
} ps_affine_f32;
ps_status ps_scan_pair_i32_f32(int exclusive, const ps_pair_i32_f32 *in, ps_pair_i32_f32 *out, size_t n,
                               void *ws, size_t ws_bytes, ps_stream_t stream);
ps_status ps_scan_affine_f32(int exclusive, const ps_affine_f32 *in, ps_affine_f32 *out, size_t n,
                             void *ws, size_t ws_bytes, ps_stream_t stream);

/*
 * Single-pass reduce-by-key and run-length encoding: the other fused
 * workloads of the decoupled look-back paper (Merrill & Garland, "Single-pass
 * Parallel Prefix Scan with Decoupled Look-back", A5 results on
 * reduce-by-key and run-length-encode).  Reduce-by-key is one scan over
 * (run count, value since the run began) pairs under the segmented-sum
 * operator -- associative, not commutative, which the method allows (section
 * 4.2: only contiguous partials are ever combined).  Run-length encoding is
 * one scan over (run count, position of the last run start) pairs: a run's
 * length is the distance from its first element to the next run's.
 *
 * A run is a maximal stretch of consecutive keys with equal bits (fp32 keys
 * compare as their 32-bit patterns: -0.0 and +0.0 are different keys, two
 * NaNs with the same bits are one).  For the j-th run, in input order:
 *     unique_keys[j] = its key,
 *     aggregates[j]  = the sum of its values (ps_reduce_by_key; int32 values
 *                      wrap modulo 2^32, fp32 values add in fp32 in an order
 *                      the caller cannot choose), or its length
 *                      (ps_run_length_encode; 32-bit unsigned count stored in
 *                      an int32 slot).
 * *num_runs (device, may be NULL) receives the number of runs m; entries m
 * and beyond of both outputs are left untouched, so each output needs room
 * for n entries when m is not known in advance.
 *
 *   key_dtype    PS_INT32, PS_INT64 or PS_FLOAT32 (keys are only compared).
 *   value_dtype  PS_INT32 or PS_FLOAT32 (ps_reduce_by_key only).
 *   keys, values device arrays of n elements (naturally aligned; 16-byte
 *                alignment of both selects the bulk-copy fast path).
 *   unique_keys  device, n entries of key_dtype; aggregates: n entries of
 *                value_dtype (int32 for run-length encoding).  Neither output
 *                may overlap an input, the other output, the workspace or
 *                num_runs (PS_ERR_OVERLAP): unlike select, reduce-by-key is
 *                not computed in place.
 *   ws           at least ps_reduce_by_key_workspace_size(key_dtype, n)
 *                bytes, 16-byte aligned, zero-filled once before first use
 *                (ps_workspace_init); the same conventions as the scans.
 *   n            below 2^32; n == 0 writes *num_runs = 0 and nothing else.
 * Errors: PS_ERR_INVALID_ARG for a bad dtype, NULL array with n > 0,
 * misaligned pointer or n >= 2^32; PS_ERR_WORKSPACE_TOO_SMALL; PS_ERR_OVERLAP;
 * PS_ERR_CUDA if the launch fails.  Device-side failures (a look-back that
 * gave up) are reported by ps_get_device_status.
 */
size_t ps_reduce_by_key_workspace_size(ps_dtype key_dtype, size_t n);
ps_status ps_reduce_by_key(ps_dtype key_dtype, ps_dtype value_dtype, const void *keys,
                           const void *values, void *unique_keys, void *aggregates,
                           uint64_t *num_runs, size_t n, void *ws, size_t ws_bytes,
                           ps_stream_t stream);
ps_status ps_run_length_encode(ps_dtype key_dtype, const void *keys, void *unique_keys,
                               int32_t *counts, uint64_t *num_runs, size_t n, void *ws,
                               size_t ws_bytes, ps_stream_t stream);

/*
 * Waits for `stream`, then reads into *out the device-side status of the
 * last call that ran a look-back kernel on `ws`: PS_OK,
 * PS_ERR_LOOKBACK_TIMEOUT, or PS_ERR_WORKSPACE_NOT_INITIALIZED (the
 * workspace was never zero-filled).  Scans of up to two tiles (see
 * ps_tile_elements) run no look-back and leave the status as it was.
 * Returns PS_ERR_CUDA if the wait or the copy fails.
 */
ps_status ps_get_device_status(const void *ws, ps_stream_t stream, ps_status *out);

/* Static, human-readable name of a status code. */
const char *ps_status_string(ps_status status);

/* cudaError_t of the last PS_ERR_CUDA returned on the calling thread. */
int ps_last_cuda_error(void);

/* Elements per tile (one CTA's share) the decoupled look-back path uses. */
size_t ps_tile_elements(ps_dtype dtype);

/*
 * Allocation-free int32 inclusive scan.  The pages have no counterpart: it
 * exists for callers that cannot allocate device memory at all -- code
 * running inside an allocator or memory-pool callback, plug-ins whose host
 * application owns every device allocation, paths that must never reach
 * the allocator -- and so cannot supply the workspace the entry points
 * above take.
 *
 * Same computation and conventions as ps_scan_inclusive_i32, except that the
 * look-back scratch lives in a fixed array inside the library's device
 * memory (PS_NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library
 * until the process exits) instead of a caller workspace.  Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - n > PS_NOALLOC_MAX_ELEMENTS returns PS_ERR_WORKSPACE_TOO_SMALL before
 *     anything is enqueued (the fixed scratch holds descriptors for at most
 *     that many elements).
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and zero-fills the
 *     array on `stream`; make that first call before any stream capture.  A
 *     failed look-up returns PS_ERR_CUDA (see ps_last_cuda_error).
 *   - All calls on a device share the one array, and each call leaves it
 *     ready for the next (as any workspace, see ps_workspace_init).  Calls
 *     whose GPU work can overlap (other streams, unordered host threads)
 *     race on it and produce wrong results; calls ordered on one stream are
 *     safe.
 *   - Every call looks the array's address up again (a host-side look-up):
 *     cudaDeviceReset destroys the loaded copy of the array, and the next
 *     call finds, and if it moved zero-fills, the new one.
 *   - There is no caller workspace to pass to ps_get_device_status; the
 *     test hook ps_testing_noalloc_scratch (prefix_scan_testing.h) gives
 *     the array's address for that.
 */
#define PS_NOALLOC_MAX_ELEMENTS 536870912u /* 2^29 elements */
#define PS_NOALLOC_SCRATCH_BYTES (256u + 72u * (PS_NOALLOC_MAX_ELEMENTS / 8192u)) /* 4.5 MiB + 256 */
ps_status ps_scan_inclusive_i32_noalloc(const int32_t *in, int32_t *out, size_t n,
                                        ps_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PREFIX_SCAN_H */
