/*
 * gc.h -- C ABI of libgc: predicate -> exclusive scan -> scatter on one
 * GB300 GPU (sm_103a).
 *
 * Operations and the passages that define them:
 *
 *   gc_exclusive_scan    out[i] = in[0] + ... + in[i-1], out[0] = 0.
 *                        "scan_2.cu -- Day 32: the work-efficient scan"
 *                        (scanExclusiveCpu, the CPU reference); the same
 *                        exclusive semantics as "compaction.cu -- Day 33"
 *                        (scanTilesExclusive, "rank[i] becomes the number of
 *                        survivors before i").
 *   gc_select_if         the elements a predicate keeps, in input order, and
 *                        their count.  "compaction.cu -- Day 33" (file
 *                        header: predicate, scan, scatter; compactCpu;
 *                        scatterCompact) and "The CUDA Handbook, ch. 13:
 *                        Stream compaction" (Listing 13-17, the single-pass
 *                        form: the highest-numbered tile writes the total).
 *   gc_partition         stable two-way partition: kept elements in input
 *                        order, then rejected ones in input order; one scan
 *                        addresses both halves through i - rank[i].
 *                        "compaction.cu -- Day 33" (partitionCpu,
 *                        scatterPartition).
 *   gc_split_radix       LSD radix sort by one-bit stable splits, bit-clear
 *                        first, one split per bit in [begin_bit, end_bit).
 *                        "CIS 565 Project 2: Stream Compaction" (radix sort
 *                        built on scan); each split is gc_partition with the
 *                        predicate "bit b is 0".
 *   gc_radix_sort        full-width stable ascending sort of int32, uint32 or
 *                        float32 keys (IEEE 754 totalOrder) by 8-bit digits,
 *                        four passes: the one-bit split generalised to a
 *                        256-way split addressed by a scan of per-tile digit
 *                        counts ("CIS 565 Project 2", radix sort built on
 *                        scan), over an order-preserving key.  The radix
 *                        passage sorts unsigned keys only; the key map is
 *                        the standard sign-flip reading of "sort by the
 *                        value" for the other two dtypes.
 *   gc_select_if_atomic  the comparison path: the same survivors and count,
 *                        placed by an atomic counter (one atomicAdd per
 *                        survivor), in no defined order.  "compaction.cu --
 *                        Day 33" (compactAtomic).  gc_select_if_atomic_tile
 *                        is the same with one atomic per tile.
 *
 * Conventions common to every entry point:
 *
 *   - Pointers named d_* are device pointers (cudaMalloc / torch memory on
 *     the current device).  Element pointers must be 4-byte aligned; 16-byte
 *     aligned element pointers take the vectorised kernels, others the same
 *     kernels with each tile staged from the 16-byte boundary below it and
 *     outputs stored element by element, with identical results.
 *   - n is an element count, 0 <= n <= GC_MAX_ELEMENTS (2^31 - 1).
 *   - Every call is asynchronous on `stream` (0 = legacy default stream):
 *     it enqueues work and returns.  Counts and totals are written to device
 *     memory on that stream; nothing is copied to the host.  The library
 *     never allocates device memory and never synchronises, except
 *     gc_query_device_status.
 *   - Scratch lives in a caller-owned workspace: d_ws, at least
 *     gc_workspace_bytes(op, n, dtype) bytes, 256-byte aligned, and
 *     zero-filled once before its first use (gc_workspace_init does that).
 *     The library leaves it valid for the next call.  One workspace must not
 *     be used by two calls that can run at the same time (different streams
 *     without ordering between them).
 *   - n == 0: the count / total outputs are set to 0, nothing else runs.
 *   - Return value: GC_OK if the work was enqueued.  Argument errors are
 *     detected on the host before anything is enqueued.  GC_ERR_CUDA means a
 *     CUDA call or launch failed (cudaGetLastError() holds the cause).
 *     Failures inside a kernel (a look-back wait that gave up) are recorded
 *     in the workspace and reported by gc_query_device_status.
 */
#ifndef GC_H
#define GC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GC_MAX_ELEMENTS 2147483647u

typedef enum {
    GC_OK = 0,
    GC_ERR_INVALID_VALUE = 1,      /* null pointer, n too large, bad enum, bad bit range, overlap */
    GC_ERR_UNSUPPORTED = 2,        /* predicate not defined for the dtype (ODD/EVEN on float32) */
    GC_ERR_WORKSPACE_TOO_SMALL = 3,
    GC_ERR_MISALIGNED = 4,         /* element pointer not 4-byte or workspace not 256-byte aligned */
    GC_ERR_CUDA = 5,               /* a CUDA runtime call or kernel launch failed */
    GC_ERR_TIMEOUT = 6,            /* device: a look-back wait gave up (see gc_query_device_status) */
    GC_ERR_DEVICE_CHECK = 7        /* device: a kernel's own bounds check refused to write */
} gc_status;

typedef enum { GC_I32 = 0, GC_U32 = 1, GC_F32 = 2 } gc_dtype;

/*
 * Predicates ("compaction.cu -- Day 33" markNonZero / markEven; "The CUDA
 * Handbook, ch. 13" isOdd):
 *   GC_PRED_NONZERO  x != 0.  For float32 the IEEE comparison: +0.0 and -0.0
 *                    are rejected, NaN, infinities and denormals are kept.
 *   GC_PRED_ODD      (x & 1) != 0, int32 / uint32 only.
 *   GC_PRED_EVEN     (x & 1) == 0, int32 / uint32 only.
 */
typedef enum { GC_PRED_NONZERO = 0, GC_PRED_ODD = 1, GC_PRED_EVEN = 2 } gc_pred;

/*
 * Parameterised predicates (gc_select_if_pred, gc_partition_pred): "The CUDA
 * Handbook, ch. 13: Stream compaction" notes that its single-pass compaction
 * "is easily modified to evaluate more-complicated predicates".
 *   GC_CMP_LT .. GC_CMP_NE   x OP operand in the dtype's own order: int32
 *                            signed, uint32 unsigned, float32 IEEE 754 (every
 *                            comparison with a NaN is false except NE; -0.0
 *                            equals +0.0).  operand is the value's 32-bit
 *                            pattern in the dtype.
 *   GC_CMP_MASK_EQ / _NE     (bits & mask) == operand / != operand on the raw
 *                            32 bits, any dtype.
 * The fixed predicates are special cases: NONZERO is NE 0, ODD is MASK_NE
 * with mask 1 and operand 0, EVEN is MASK_EQ with mask 1 and operand 0.
 */
typedef enum {
    GC_CMP_LT = 0,
    GC_CMP_LE = 1,
    GC_CMP_GT = 2,
    GC_CMP_GE = 3,
    GC_CMP_EQ = 4,
    GC_CMP_NE = 5,
    GC_CMP_MASK_EQ = 6,
    GC_CMP_MASK_NE = 7
} gc_cmp;

typedef struct {
    gc_cmp cmp;
    uint32_t operand; /* the operand's bits (LT..NE) or the masked value (MASK_*) */
    uint32_t mask;    /* MASK_* only */
} gc_predicate;

typedef enum {
    GC_OP_EXCLUSIVE_SCAN = 0,
    GC_OP_SELECT_IF = 1,
    GC_OP_PARTITION = 2,
    GC_OP_SPLIT_RADIX = 3,
    GC_OP_SELECT_IF_ATOMIC = 4,
    GC_OP_INCLUSIVE_SCAN = 5,
    GC_OP_RADIX_SORT = 6,
    GC_OP_REDUCE = 7,      /* gc_reduce */
    GC_OP_COUNT_IF = 8     /* gc_count_if */
} gc_op;

/* Static, never NULL, "unknown status" for values outside the enum. */
const char *gc_status_string(gc_status status);

/* Library version string, static. */
const char *gc_version(void);

/*
 * Workspace bytes op needs for n elements of dtype (dtype is ignored for
 * GC_OP_SPLIT_RADIX, whose keys and payloads are uint32; GC_OP_RADIX_SORT
 * needs the same bytes for every dtype).  Returns 0 for an
 * unknown op or dtype or n > GC_MAX_ELEMENTS.  A workspace sized for the
 * largest (op, n) it will serve can be reused by every smaller call.
 */
size_t gc_workspace_bytes(gc_op op, size_t n, gc_dtype dtype);

/*
 * Elements per tile of op's kernel (one CTA's share of the input): a size
 * that is a multiple of it fills every tile, other sizes leave a ragged last
 * tile.  Returns 0 for an unknown op.
 */
size_t gc_tile_elements(gc_op op);

/* cudaMemsetAsync(d_ws, 0, ws_bytes, stream): prepares a new workspace. */
gc_status gc_workspace_init(void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Exclusive scan.  d_in and d_out hold n elements of dtype; d_in == d_out
 * (in place) is allowed, any other overlap is GC_ERR_INVALID_VALUE.
 * d_total (nullable) receives in[0] + ... + in[n-1] as one element of dtype.
 * int32 and uint32 add modulo 2^32 (the same bits).  float32 adds within a
 * tile in float32 with round-to-nearest and carries the running prefix
 * between tiles as an unevaluated pair of float32 values (about 48
 * significant bits; the one-tile-per-CTA kernel run when the device
 * refuses a cooperative grid carries a float64); the sums of the tiles between a CTA's consecutive
 * tiles are added in float32.  Each output is the prefix of its 4-element
 * vector, rounded to float32, plus the sum of the vector's earlier elements,
 * so the result is within a few float32 roundings of the exact prefix
 * (relative error below 1e-6 for non-negative inputs); the summation order
 * is not sequential.
 */
gc_status gc_exclusive_scan(const void *d_in, void *d_out, void *d_total,
                            size_t n, gc_dtype dtype, void *d_ws,
                            size_t ws_bytes, cudaStream_t stream);

/*
 * Inclusive scan: out[i] = in[0] + ... + in[i] (the inclusive scans of
 * "scan.cu -- Day 31: prefix sum (scan), part 1", whole-array rather than
 * per block).  Everything else as gc_exclusive_scan, including in-place
 * operation and d_total.  Workspace: gc_workspace_bytes(GC_OP_INCLUSIVE_SCAN,
 * ...), the same as the exclusive scan's.
 */
gc_status gc_inclusive_scan(const void *d_in, void *d_out, void *d_total,
                            size_t n, gc_dtype dtype, void *d_ws,
                            size_t ws_bytes, cudaStream_t stream);

/*
 * Stable select-if.  d_out must have room for n elements (the worst case);
 * elements [0, *d_count) are the survivors in input order, the rest of d_out
 * is untouched.  *d_count is written by the kernel (a uint32 in device
 * memory).  d_in and d_out must not overlap.
 */
gc_status gc_select_if(const void *d_in, void *d_out, uint32_t *d_count,
                       size_t n, gc_dtype dtype, gc_pred pred, void *d_ws,
                       size_t ws_bytes, cudaStream_t stream);

/*
 * Stable partition.  d_out (n elements) receives the predicate-true
 * elements in input order followed by the false ones in input order;
 * *d_count_true (device uint32) is the size of the first half.  d_in and
 * d_out must not overlap.  Two kernels: a count of the true elements, then
 * one pass that scans and scatters both halves.
 */
gc_status gc_partition(const void *d_in, void *d_out, uint32_t *d_count_true,
                       size_t n, gc_dtype dtype, gc_pred pred, void *d_ws,
                       size_t ws_bytes, cudaStream_t stream);

/*
 * gc_select_if and gc_partition with a parameterised predicate.  `pred` is a
 * host pointer, read during the call.  GC_ERR_INVALID_VALUE for a NULL pred
 * or an unknown cmp; otherwise the conventions, workspace
 * (GC_OP_SELECT_IF / GC_OP_PARTITION) and errors of the fixed-predicate
 * entry points.
 */
gc_status gc_select_if_pred(const void *d_in, void *d_out, uint32_t *d_count,
                            size_t n, gc_dtype dtype, const gc_predicate *pred,
                            void *d_ws, size_t ws_bytes, cudaStream_t stream);
gc_status gc_partition_pred(const void *d_in, void *d_out, uint32_t *d_count_true,
                            size_t n, gc_dtype dtype, const gc_predicate *pred,
                            void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * LSD radix sort by one-bit stable splits over bits [begin_bit, end_bit),
 * 0 <= begin_bit <= end_bit <= 32, lowest bit first, keys with the bit clear
 * first.  With [0, 32) the keys come out ascending, equal keys in input
 * order, and d_vals_out holds the payloads permuted with them.  d_vals_in
 * and d_vals_out are both NULL (keys only) or both non-NULL.  The result
 * always lands in d_keys_out / d_vals_out; the intermediate ping-pong
 * buffers live in the workspace.  An input may equal its output (in place);
 * any other overlap between the four arrays is GC_ERR_INVALID_VALUE.  An
 * empty bit range copies.  One histogram kernel, then one split kernel per
 * bit.
 */
gc_status gc_split_radix(const uint32_t *d_keys_in, const uint32_t *d_vals_in,
                         uint32_t *d_keys_out, uint32_t *d_vals_out, size_t n,
                         int begin_bit, int end_bit, void *d_ws,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * Stable ascending radix sort of n keys of dtype, payloads carried: int32 in
 * signed order, uint32 in unsigned order, float32 in IEEE 754 totalOrder
 * (-NaN < -inf < negatives < -0 < +0 < positives < +inf < +NaN; NaNs by
 * payload bits, as patterns).  Equal keys keep their input order.  The
 * sort runs four stable passes over the 8-bit digits, lowest first, of the
 * order-preserving key k(x) = x ^ (signfill(x) & neg) ^ flip (int32: neg 0,
 * flip 2^31; float32: neg 2^31 - 1, flip 2^31; uint32: both 0); each pass
 * is three launches (digit counts per 4096-key tile, one scan of the
 * counts, the scatter).  The keys are moved as they are, never rewritten,
 * so d_keys_out holds the input's own bit patterns.  The same array and
 * aliasing rules as gc_split_radix: keys and payloads both or keys alone,
 * an input may equal its output, no other overlap.  The workspace,
 * gc_workspace_bytes(GC_OP_RADIX_SORT, n, dtype), holds the ping-pong
 * buffers and a table of 256 counts per tile.  Keys are d_keys_in /
 * d_keys_out as void * to any of the three dtypes, 4-byte aligned.
 */
gc_status gc_radix_sort(const void *d_keys_in, const uint32_t *d_vals_in,
                        void *d_keys_out, uint32_t *d_vals_out, size_t n,
                        gc_dtype dtype, void *d_ws, size_t ws_bytes,
                        cudaStream_t stream);

/*
 * The atomic-counter comparison path of "compaction.cu -- Day 33"
 * (compactAtomic): every survivor takes its output slot with one atomicAdd
 * on the single counter *d_count and is written there.  The same survivors
 * and the same *d_count as gc_select_if, in an order the hardware decides:
 * only the multiset of d_out[0, *d_count) is defined.  Its cost grows with
 * the number of survivors, all of which serialise on one address.  The
 * counter is cleared on the stream before the kernel; the workspace
 * (gc_workspace_bytes(GC_OP_SELECT_IF_ATOMIC, ...)) is checked but unused.
 */
gc_status gc_select_if_atomic(const void *d_in, void *d_out, uint32_t *d_count,
                              size_t n, gc_dtype dtype, gc_pred pred,
                              void *d_ws, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * gc_select_if_atomic with one atomic per tile of
 * gc_tile_elements(GC_OP_SELECT_IF_ATOMIC) elements instead of one per
 * survivor: each CTA ranks its tile's survivors, claims a run of that many
 * slots with one atomicAdd on *d_count and writes the run.  Survivors keep
 * their input order within a tile; the tiles' runs land in the order their
 * atomics resolve.  Same arguments, workspace and output contract as
 * gc_select_if_atomic.  Not on the pages: it shows how much of the
 * comparator's cost is the one-address serialisation.
 */
gc_status gc_select_if_atomic_tile(const void *d_in, void *d_out, uint32_t *d_count,
                                   size_t n, gc_dtype dtype, gc_pred pred,
                                   void *d_ws, size_t ws_bytes,
                                   cudaStream_t stream);

/*
 * gc_select_if without a workspace, for callers that cannot allocate device
 * memory where they need the compaction: a plugin whose host framework owns
 * the device memory budget and forbids allocations behind its back, or a
 * latency-critical loop that must not pay for cudaMalloc / cudaFree, which
 * may synchronise the device.  There is no counterpart on the pages this
 * library follows; the result is exactly gc_select_if's.
 *
 * The scratch the kernels need lives in one file-scope device array of
 * 1,049,600 bytes inside the library, held by every GPU that loads it until
 * the process exits; it serves n <= GC_NOALLOC_MAX_ELEMENTS (2^28), and
 * larger n returns GC_ERR_INVALID_VALUE.  The first call on a device (with
 * that device current) looks up the array's device address and caches it;
 * make that first call before any stream capture begins.  Every call shares
 * the array: each clears what must start at zero on its own stream, and
 * calls that can overlap on the GPU (different streams with no ordering
 * between them) race on it.  Device-side failures of this entry point (a
 * bounded wait that gave up, a refused store) are recorded in that array and
 * reported by gc_select_if_noalloc_status.  The cached address belongs to
 * the device's primary context: after a cudaDeviceReset the array and the
 * cache are gone, and the library must not be called again in that process.
 * No allocation of any kind.
 */
#define GC_NOALLOC_MAX_ELEMENTS 268435456u
gc_status gc_select_if_noalloc(const void *d_in, void *d_out, uint32_t *d_count,
                               size_t n, gc_dtype dtype, gc_pred pred,
                               cudaStream_t stream);

/*
 * SYNCHRONOUS.  gc_query_device_status for the fixed array of
 * gc_select_if_noalloc on the current device: waits for `stream`, reads and
 * clears the array's error word, and after an error also resets its start
 * barrier, which a barrier wait that gave up leaves marked (so that later
 * calls time out instead of passing it early).  Returns GC_OK,
 * GC_ERR_TIMEOUT or GC_ERR_DEVICE_CHECK (the outputs of the failed call are
 * undefined), or GC_ERR_CUDA.  Like the entry point it allocates nothing.
 */
gc_status gc_select_if_noalloc_status(cudaStream_t stream);

/*
 * ---------------------------------------------------------------- shards
 *
 * A scan, select-if or partition of one array cut into P contiguous shards
 * (one per GPU, each in its own memory, or several on one GPU), computed
 * shard by shard.  Each shard needs only what the shards before it
 * contribute: the sum of their elements (scan), the number of survivors
 * before it (select-if), and for partition also the total number kept, T,
 * since rejected elements start at T.  That is the decoupled look-back of
 * "The CUDA Handbook, ch. 13: Stream compaction" one level up, tiles
 * becoming shards, and the kept / rejected addressing rank[i] and
 * T + i - rank[i] of "compaction.cu -- Day 33" (scatterPartition).
 *
 * Sequence on rank r, all on one stream, nothing read back to the host:
 *   1. pre-pass: gc_reduce (scan) or gc_count_if (select-if, partition)
 *      writes this shard's total into slot r of a device array of P words;
 *   2. exchange: every rank gathers the P words (an all-gather, e.g. NCCL;
 *      on one GPU the P slots are simply written in place);
 *   3. gc_shard_offsets computes rank r's offsets from the P words;
 *   4. the placed pass: gc_exclusive_scan_carry, gc_select_if_at or
 *      gc_partition_at.
 * Every placed pass reads the input once more (4 B per element), so a
 * sharded scan moves 12 B per element and a sharded select-if 8 + 4 * kept.
 */
#define GC_MAX_SHARDS 65536u

/*
 * d_total (one element of dtype) = in[0] + ... + in[n-1]: int32 / uint32
 * modulo 2^32, float32 summed in float pairs per thread and in double across
 * CTAs, rounded once (deterministic for a given device).  Workspace:
 * gc_workspace_bytes(GC_OP_REDUCE, n, dtype).  n == 0 writes 0.
 */
gc_status gc_reduce(const void *d_in, void *d_total, size_t n, gc_dtype dtype, void *d_ws,
                    size_t ws_bytes, cudaStream_t stream);

/*
 * *d_count = how many of the n elements pred keeps (the count pre-pass of
 * gc_partition alone).  Workspace: gc_workspace_bytes(GC_OP_COUNT_IF, ...).
 * Errors as gc_select_if.
 */
gc_status gc_count_if(const void *d_in, uint32_t *d_count, size_t n, gc_dtype dtype,
                      gc_pred pred, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Offsets of shard `rank` of `parts` (device writes, one thread):
 *   op GC_OP_EXCLUSIVE_SCAN: d_totals = parts elements of dtype (the shards'
 *       gc_reduce totals); d_offsets receives one element of dtype, the sum
 *       of totals [0, rank) (int modulo 2^32; float32 summed in double).
 *   op GC_OP_SELECT_IF: d_totals = parts uint32 counts; d_offsets receives
 *       one uint64 (8-byte aligned), the sum of counts [0, rank).
 *   op GC_OP_PARTITION: as select-if, plus h_sizes (host, parts element
 *       counts, read during the call); d_offsets receives two uint64: kept
 *       before = counts [0, rank) summed, and the first rejected position
 *       T + (h_sizes [0, rank) summed) - kept before, T = all counts summed.
 * h_sizes is ignored except for partition.  Errors: GC_ERR_INVALID_VALUE for
 * another op, a bad dtype, parts == 0 or > GC_MAX_SHARDS, rank >= parts,
 * NULL pointers or a size > GC_MAX_ELEMENTS; GC_ERR_MISALIGNED.
 */
gc_status gc_shard_offsets(gc_op op, gc_dtype dtype, const uint32_t *d_totals,
                           const uint64_t *h_sizes, size_t parts, size_t rank, void *d_offsets,
                           cudaStream_t stream);

/*
 * gc_exclusive_scan plus a carry-in: out[i] = *d_carry + in[0] + ... +
 * in[i-1], and d_total (nullable) = *d_carry + the sum of all n, i.e. the
 * carry of the shard after this one.  d_carry is one device element of
 * dtype, read by the kernel (non-NULL).  Same workspace, precision, in-place
 * rule and errors as gc_exclusive_scan; n == 0 copies the carry to d_total.
 */
gc_status gc_exclusive_scan_carry(const void *d_in, void *d_out, void *d_total, size_t n,
                                  gc_dtype dtype, const void *d_carry, void *d_ws,
                                  size_t ws_bytes, cudaStream_t stream);

/*
 * gc_select_if whose survivors go to d_out[*d_base + rank] instead of
 * d_out[rank]: d_out is the whole output (out_capacity elements, in this
 * device's memory) and *d_base (device uint64, 8-byte aligned) the number
 * of survivors of the shards before this one.  *d_count receives this
 * shard's own count.  A run that would end past out_capacity is not written
 * and is reported as GC_ERR_DEVICE_CHECK by gc_query_device_status.
 * Workspace and errors as gc_select_if.
 */
gc_status gc_select_if_at(const void *d_in, void *d_out, size_t out_capacity,
                          const uint64_t *d_base, uint32_t *d_count, size_t n, gc_dtype dtype,
                          gc_pred pred, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * gc_partition of one shard into the whole output: kept elements to
 * d_out[d_offsets[0] + rank[i]], rejected ones to d_out[d_offsets[1] + i -
 * rank[i]] (the two uint64 of gc_shard_offsets), so that the shards together
 * write the stable partition of the whole array.  One pass, no count
 * pre-pass (T is in the offsets).  *d_count_true receives this shard's kept
 * count.  out_capacity >= n; runs past it are refused as in gc_select_if_at.
 * Workspace and errors as gc_partition.
 */
gc_status gc_partition_at(const void *d_in, void *d_out, size_t out_capacity,
                          const uint64_t *d_offsets, uint32_t *d_count_true, size_t n,
                          gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * SYNCHRONOUS.  Waits for `stream`, then reads and clears the device-side
 * error word of the workspace.  Returns GC_OK, GC_ERR_TIMEOUT if a kernel's
 * bounded wait (a look-back, a staged load, or the start barrier at which a
 * persistent kernel's CTAs meet after clearing their status words) gave up
 * since the last query, GC_ERR_DEVICE_CHECK if a kernel found an output range
 * outside its buffer (a corrupted workspace) and skipped those stores -- in
 * both cases the outputs of that call are undefined -- or GC_ERR_CUDA if the
 * synchronisation itself failed.  After an error it also resets the start
 * barrier's arrival counter, which a barrier wait that gave up leaves marked
 * so that later calls time out rather than pass the barrier early.
 */
gc_status gc_query_device_status(void *d_ws, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GC_H */
