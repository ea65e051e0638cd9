/*
 * gc_testing.h -- test hooks of libgc.  Not for production callers.
 *
 * They exist so that the library's failure handling can be exercised on a
 * real GPU without faulting it: every wait inside a kernel has a time limit
 * after which the kernel records GC_ERR_TIMEOUT in the workspace and
 * finishes normally, and this hook makes one wait run out on purpose.
 */
#ifndef GC_TESTING_H
#define GC_TESTING_H

#include "gc.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gc_select_if with a planted failure: tile 0 is never taken by any CTA, so
 * tile 1's look-back waits for a status word that nobody writes, gives up
 * after timeout_ns nanoseconds of device time, records GC_ERR_TIMEOUT in the
 * workspace error word and lets its successors finish.  Requires at least two
 * tiles (n > gc_tile_elements(GC_OP_SELECT_IF)).  The output is undefined;
 * gc_query_device_status then returns GC_ERR_TIMEOUT, and the workspace is
 * fit for the next call.
 */
gc_status gc_testing_select_if_skip_tile0(const void *d_in, void *d_out, uint32_t *d_count,
                                          size_t n, gc_dtype dtype, gc_pred pred, void *d_ws,
                                          size_t ws_bytes, uint64_t timeout_ns,
                                          cudaStream_t stream);

/*
 * gc_exclusive_scan with a stalled start barrier.  A persistent kernel clears
 * its own status words and then waits at a start barrier in the workspace
 * header until every CTA has arrived; this hook first marks the barrier's
 * arrival counter the way a barrier wait that ran out leaves it, so no CTA
 * of this call ever sees the barrier complete.  Each CTA's wait gives up
 * after timeout_ns nanoseconds of device time, records GC_ERR_TIMEOUT and
 * carries on.  Requires a 16-byte-aligned d_in and n >= 1; otherwise GC_ERR_INVALID_VALUE, and argument errors as
 * gc_exclusive_scan.  The output is undefined; gc_query_device_status then
 * returns GC_ERR_TIMEOUT and clears the barrier's words, after which the
 * workspace is fit for the next call.
 */
gc_status gc_testing_exclusive_scan_stalled_barrier(const void *d_in, void *d_out, void *d_total,
                                                    size_t n, gc_dtype dtype, void *d_ws,
                                                    size_t ws_bytes, uint64_t timeout_ns,
                                                    cudaStream_t stream);

/*
 * gc_select_if_noalloc with a stalled start barrier: the fixed array's
 * arrival counter is marked as a barrier wait that ran out leaves it, so
 * every CTA's barrier wait gives up after timeout_ns, records GC_ERR_TIMEOUT
 * and carries on.  Requires a 16-byte-aligned d_in and n >= 1 (otherwise
 * GC_ERR_INVALID_VALUE), else the argument errors of gc_select_if_noalloc.
 * The output is undefined; gc_select_if_noalloc_status then returns
 * GC_ERR_TIMEOUT and clears the barrier.
 */
gc_status gc_testing_select_if_noalloc_stalled_barrier(const void *d_in, void *d_out,
                                                       uint32_t *d_count, size_t n,
                                                       gc_dtype dtype, gc_pred pred,
                                                       uint64_t timeout_ns,
                                                       cudaStream_t stream);

/*
 * Process-wide switch: while on is non-zero, every scan, select-if and
 * partition (the one-bit split included) runs its one-tile-per-CTA kernels
 * (dynamic tile ids, a warp look-back, a memset of the tile counter and
 * status words first), which otherwise run only when the device refuses a
 * cooperative grid.  The results are the same; tests use it to keep those
 * kernels covered.  Not thread-safe with respect to calls in flight on other
 * host threads.
 */
void gc_testing_force_fallback(int on);

#ifdef __cplusplus
}
#endif

#endif /* GC_TESTING_H */
