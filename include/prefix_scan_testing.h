/*
 * prefix_scan_testing.h -- test hooks of the prefix-scan library.
 *
 * These entry points expose one internal piece of the single-pass scan, the
 * warp-parallel decoupled look-back ("Single-pass Parallel Prefix Scan with
 * Decoupled Look-back", summary page, sections 4.1 and 4.4), so that it can
 * be checked alone on hand-made tile status descriptors -- e.g. the
 * execution snapshot of Figure 6 (section 4.3) -- and so that its bounded
 * wait can be made to run out (a descriptor that nothing ever publishes)
 * without faulting or hanging the GPU.  They are not needed to compute a
 * scan.  Conventions (device pointers, stream, errors) are those of
 * prefix_scan.h.
 */
#ifndef PREFIX_SCAN_TESTING_H
#define PREFIX_SCAN_TESTING_H

#include "prefix_scan.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Descriptor status flags: nothing published / aggregate / inclusive prefix. */
enum { PS_FLAG_X = 0, PS_FLAG_A = 1, PS_FLAG_P = 2 };

/* Size in bytes of one tile status descriptor for `dtype` (8 or 16). */
size_t ps_testing_descriptor_bytes(ps_dtype dtype);

/*
 * Host-side encoding of one descriptor of call `epoch` (< 2^30): writes
 * the first 8 bytes (16 for int64) of a ps_testing_descriptor_bytes-byte
 * slot to `out` (host memory), holding `flag`, `epoch` and the value at
 * `value` (host pointer to one element of `dtype`).  PS_ERR_INVALID_ARG on
 * a bad dtype, flag, epoch or NULL pointer.
 */
ps_status ps_testing_encode_descriptor(ps_dtype dtype, int flag, uint32_t epoch, const void *value,
                                       void *out);

/*
 * Runs the look-back of tile `tile` (>= 1) of call `epoch` with one warp
 * over the device array `desc` of at least `tile` descriptor slots, polling
 * at most `max_polls` times.  Writes the exclusive prefix (one element of
 * `dtype`) to device `result`; `status` (device, one uint64, caller-zeroed)
 * receives epoch << 8 | PS_ERR_LOOKBACK_TIMEOUT if the wait ran out.  Only
 * descriptors 0 .. tile-1 are read; descriptors of another epoch count as
 * not published.  Asynchronous on `stream`.
 */
ps_status ps_testing_lookback(ps_dtype dtype, const void *desc, int64_t tile, uint32_t epoch,
                              uint32_t max_polls, void *result, uint64_t *status,
                              ps_stream_t stream);

/*
 * The call number (epoch, modulo 2^30) the next scan on `ws` will run as:
 * read after waiting for `stream`, or set (marking the workspace as in
 * use), so that a test can bring a workspace to the epoch wrap-around
 * without 2^30 calls.
 */
ps_status ps_testing_workspace_epoch(const void *ws, ps_stream_t stream, uint32_t *epoch);
ps_status ps_testing_set_workspace_epoch(void *ws, uint32_t epoch, ps_stream_t stream);

/*
 * The device address (for the current device) of the fixed scratch array
 * that ps_scan_inclusive_i32_noalloc uses in place of a workspace, written
 * to *scratch, so that a test can read the status of the last such call
 * with ps_get_device_status(*scratch, ...).  Does the same set-up as a
 * first ps_scan_inclusive_i32_noalloc call on the device (the zero-fill is
 * enqueued on `stream`).  PS_ERR_CUDA if the look-up fails.
 */
ps_status ps_testing_noalloc_scratch(void **scratch, ps_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PREFIX_SCAN_TESTING_H */
