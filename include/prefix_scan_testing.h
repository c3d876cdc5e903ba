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
 * Host-side encoding of one descriptor: writes ps_testing_descriptor_bytes
 * bytes to `out` (host memory) holding `flag` and the value at `value`
 * (host pointer to one element of `dtype`).  PS_ERR_INVALID_ARG on a bad
 * dtype, flag or NULL pointer.
 */
ps_status ps_testing_encode_descriptor(ps_dtype dtype, int flag, const void *value, void *out);

/*
 * Runs the look-back of tile `tile` (>= 1) with one warp over the device
 * array `desc` of at least `tile` descriptors, polling at most `max_polls`
 * times.  Writes the exclusive prefix (one element of `dtype`) to device
 * `result`; `status` (device, one uint32, caller-zeroed) receives
 * PS_ERR_LOOKBACK_TIMEOUT if the wait ran out.  Only descriptors
 * 0 .. tile-1 are read.  Asynchronous on `stream`.
 */
ps_status ps_testing_lookback(ps_dtype dtype, const void *desc, int64_t tile, uint32_t max_polls,
                              void *result, uint32_t *status, ps_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PREFIX_SCAN_TESTING_H */
