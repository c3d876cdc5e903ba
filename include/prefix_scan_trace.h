/*
 * prefix_scan_trace.h -- the pipeline trace of the persistent single-pass
 * kernels: the scan, select / partition, reduce-by-key and run-length
 * encoding.
 *
 * The decoupled look-back ("Single-pass Parallel Prefix Scan with Decoupled
 * Look-back", summary page, sections 4.1 and 4.4) hides the look-back's
 * latency only while each tile's aggregate (A) and inclusive prefix (P)
 * appear soon enough; the trace shows where a tile's time goes.  A build of
 * the library with PS_TRACE defined records, for each of the first
 * ps_trace_capacity() tiles of every launch of each of those kernels (the
 * kernel's last launch overwrites; each kernel keeps its own record), the
 * GPU's global nanosecond timer at the points below, the CTA that claimed
 * the tile, and the windows its look-back walked and the re-polls of
 * unpublished descriptors it made.  The product build records
 * nothing: ps_trace_capacity() returns 0 and ps_trace_read fails.
 */
#ifndef PREFIX_SCAN_TRACE_H
#define PREFIX_SCAN_TRACE_H

#include "prefix_scan.h"

/* Trace points, in pipeline order (index into a tile's PS_TRACE_POINTS). */
#define PS_TRACE_CLAIM 0             /* tile id taken from the counter (a1) */
#define PS_TRACE_DATA 1              /* tile landed in shared memory (a2) */
#define PS_TRACE_AGGREGATE 2         /* A (tile 0: P) published (a6) */
#define PS_TRACE_LOOKBACK_START 3    /* look-back warp starts on the tile (a7) */
#define PS_TRACE_PREFIX 4            /* P published, prefix handed over (a8) */
#define PS_TRACE_COMPUTE_START 5     /* compute warps start on the tile (a3) */
#define PS_TRACE_PREFIX_RECEIVED 6   /* compute warps have the prefix (a9) */
#define PS_TRACE_STORED 7            /* compute warp 0 issued its stores (a9) */
#define PS_TRACE_POINTS 8
#ifndef PS_TRACE_TILES
#define PS_TRACE_TILES 65536
#endif
/* Per-CTA trace points (index into a CTA's PS_TRACE_CTA_POINTS). */
#define PS_TRACE_CTA_ENTRY 0         /* thread 0 starts */
#define PS_TRACE_CTA_HEADER 1        /* the CTA has the workspace header's verdict */
#define PS_TRACE_CTA_DONE 2          /* compute warp 0 leaves its loop */
#define PS_TRACE_CTA_POINTS 3
#ifndef PS_TRACE_CTAS
#define PS_TRACE_CTAS 1024
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Which kernel's record to read. */
#define PS_TRACE_KERNEL_SCAN 0       /* persistent scan (ps_scan and its relatives) */
#define PS_TRACE_KERNEL_SELECT 1     /* select and partition */
#define PS_TRACE_KERNEL_RBK 2        /* reduce-by-key */
#define PS_TRACE_KERNEL_RLE 3        /* run-length encoding */

/* Tiles a trace holds; 0 when this build records none. */
size_t ps_trace_capacity(void);

/*
 * Waits for the device, then copies the trace of the first `tiles` tiles
 * (<= ps_trace_capacity()) of the last launch of `kernel` (a
 * PS_TRACE_KERNEL_* value) to host memory: timestamps[t * PS_TRACE_POINTS
 * + k] (ns), lookback[t] (windows walked << 16 | re-polls, each saturating at 65535; tile 0 and tiles
 * whose look-back did not run keep old values), cta[t].  Entries of tiles
 * the launch did not reach keep older values.  The points a kernel does not
 * pass keep older values too (reduce-by-key and run-length encoding record
 * the stores of their compute warp 0 at STORED).  PS_ERR_INVALID_ARG in a
 * build without the trace or for bad arguments; PS_ERR_CUDA if a copy
 * fails.
 */
ps_status ps_trace_read(int kernel, uint64_t *timestamps, uint32_t *lookback, int32_t *cta, size_t tiles);

/*
 * The same for the CTAs of the last launch: timestamps[c *
 * PS_TRACE_CTA_POINTS + k] (ns) for the first `ctas` (<= PS_TRACE_CTAS)
 * CTAs.  Same errors as ps_trace_read.
 */
ps_status ps_trace_read_ctas(int kernel, uint64_t *timestamps, size_t ctas);

#ifdef __cplusplus
}
#endif

#endif /* PREFIX_SCAN_TRACE_H */
