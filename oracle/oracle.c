/*
 * oracle.c -- the plain CPU oracle for the predicate -> exclusive scan ->
 * scatter path (stream compaction, stable partition, one-bit LSD radix sort,
 * and the exclusive scan on its own).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check in __graft_entry__.py and the CPU-baseline leg of bench.py may load
 * this library.  The CUDA library never calls it, links it or includes
 * anything from it, and this file includes nothing from the CUDA library.
 *
 * Every function is the plain definition of the result, written as one
 * sequential loop over the input: no tiles, no blocking, no threads, no
 * intrinsics.  Where the method reaches exactly the same result faster, the
 * oracle is that definition.  Sources, by page:
 *
 *   [Day 33]  "compaction.cu -- Day 33: stream compaction and partition, by
 *             predicate, scan and scatter" (file header; compactCpu;
 *             partitionCpu; scatterPartition; compactAtomic)
 *   [Day 32]  "scan_2.cu -- Day 32: the work-efficient scan" (CPU reference
 *             scanExclusiveCpu, which accumulates in double)
 *   [Handbook 13] "The CUDA Handbook, ch. 13: Stream compaction"
 *             (Listing 13-17, isOdd and the single-pass compaction)
 *   [CIS 565] "CIS 565 Project 2: Stream Compaction" (radix sort section)
 *
 * Elements travel as raw 32-bit patterns (uint32_t); the dtype argument says
 * how the predicate reads them.  Integer scans wrap modulo 2^32, which is the
 * same bit pattern for int32 and uint32.  The float scan accumulates in
 * double, as the Day 32 CPU reference does, and returns the double prefixes
 * so that a caller can compare a float32 result against them.
 *
 * Nothing here allocates except orc_split_radix, which needs one scratch
 * pair for its ping-pong, and returns -1 if malloc fails.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Numbering shared with the Python wrapper (oracle/__init__.py). */
enum { ORC_I32 = 0, ORC_U32 = 1, ORC_F32 = 2 };
enum { ORC_NONZERO = 0, ORC_ODD = 1, ORC_EVEN = 2 };

static float bits_to_float(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/*
 * 1 if the predicate is defined for this dtype, 0 if not.  Odd and even are
 * bit tests on an integer ([Handbook 13], isOdd: x & 1) and have no meaning
 * for a float, so they are unsupported there.
 */
int orc_pred_supported(int dtype, int pred)
{
    if (dtype != ORC_I32 && dtype != ORC_U32 && dtype != ORC_F32) return 0;
    if (pred == ORC_NONZERO) return 1;
    if (pred == ORC_ODD || pred == ORC_EVEN) return dtype != ORC_F32;
    return 0;
}

/*
 * The predicate, one element at a time.
 *   NONZERO  x != 0         ([Day 33], markNonZero / compactCpu).  For float
 *                           the comparison is IEEE: -0.0 equals 0 and is
 *                           dropped, NaN differs from 0 and is kept.
 *   ODD      (x & 1) != 0   ([Handbook 13], isOdd).  Two's complement makes
 *                           this right for negative int32 as well.
 *   EVEN     (x & 1) == 0   ([Day 33], markEven / partitionCpu).
 */
static int keep(uint32_t bits, int dtype, int pred)
{
    if (pred == ORC_NONZERO) {
        if (dtype == ORC_F32) return bits_to_float(bits) != 0.0f;
        return bits != 0u;
    }
    if (pred == ORC_ODD) return (bits & 1u) != 0u;
    return (bits & 1u) == 0u; /* ORC_EVEN */
}

/* Number of elements the predicate keeps. */
size_t orc_count_if(const uint32_t *in, size_t n, int dtype, int pred)
{
    size_t c = 0;
    for (size_t i = 0; i < n; ++i) c += (size_t)keep(in[i], dtype, pred);
    return c;
}

/*
 * Exclusive scan over int32 or uint32 bit patterns: out[0] = 0 and
 * out[i] = in[0] + ... + in[i-1], every add modulo 2^32.  Returns the total
 * in[0] + ... + in[n-1] (the "top of the scan", [Day 33] launchScan).
 * out may equal in: each in[i] is read before out[i] is written.
 */
uint32_t orc_exclusive_scan_u32(const uint32_t *in, uint32_t *out, size_t n)
{
    uint32_t running = 0u;
    for (size_t i = 0; i < n; ++i) {
        const uint32_t v = in[i];
        out[i] = running;
        running += v;
    }
    return running;
}

/*
 * Exclusive scan of float32 inputs with a double accumulator, returned as
 * double ([Day 32] scanExclusiveCpu, minus its final cast to float).  With
 * inputs that are multiples of 2^-24 and totals below 2^29 every prefix is
 * exact in double.
 */
double orc_exclusive_scan_f32(const float *in, double *out, size_t n)
{
    double running = 0.0;
    for (size_t i = 0; i < n; ++i) {
        out[i] = running;
        running += (double)in[i];
    }
    return running;
}

/*
 * Inclusive scan, the same loops with the element added before it is
 * stored.  Kept beside the exclusive forms because inclusive = exclusive
 * shifted by one, which the tests use as a cross-check.
 */
uint32_t orc_inclusive_scan_u32(const uint32_t *in, uint32_t *out, size_t n)
{
    uint32_t running = 0u;
    for (size_t i = 0; i < n; ++i) {
        running += in[i];
        out[i] = running;
    }
    return running;
}

double orc_inclusive_scan_f32(const float *in, double *out, size_t n)
{
    double running = 0.0;
    for (size_t i = 0; i < n; ++i) {
        running += (double)in[i];
        out[i] = running;
    }
    return running;
}

/*
 * Stable select-if: the elements the predicate keeps, in input order.
 * Returns how many were kept ([Day 33] compactCpu; [Handbook 13] Listing
 * 13-17 computes the same function in one pass).  out needs room for n.
 */
size_t orc_select_if(const uint32_t *in, uint32_t *out, size_t n, int dtype,
                     int pred)
{
    size_t m = 0;
    for (size_t i = 0; i < n; ++i) {
        if (keep(in[i], dtype, pred)) {
            out[m] = in[i];
            ++m;
        }
    }
    return m;
}

/*
 * Stable two-way partition: every element the predicate keeps, in input
 * order, then every element it rejects, in input order.  Two passes, one per
 * half, exactly as [Day 33] partitionCpu does.  Returns the size of the first
 * half.  out needs room for n.
 */
size_t orc_partition(const uint32_t *in, uint32_t *out, size_t n, int dtype,
                     int pred)
{
    size_t first = 0;
    for (size_t i = 0; i < n; ++i) {
        if (keep(in[i], dtype, pred)) {
            out[first] = in[i];
            ++first;
        }
    }
    size_t second = first;
    for (size_t i = 0; i < n; ++i) {
        if (!keep(in[i], dtype, pred)) {
            out[second] = in[i];
            ++second;
        }
    }
    return first;
}

/*
 * One stable split by bit b, bit-clear first, carrying an optional payload.
 * This is the stable partition above with the predicate "bit b of the key is
 * 0", the step a one-bit LSD radix sort repeats once per bit.  Returns the
 * number of keys with the bit clear.
 */
static size_t split_by_bit(const uint32_t *keys, const uint32_t *vals,
                           uint32_t *keys_out, uint32_t *vals_out, size_t n,
                           int b)
{
    size_t zeros = 0;
    for (size_t i = 0; i < n; ++i) {
        if (((keys[i] >> b) & 1u) == 0u) {
            keys_out[zeros] = keys[i];
            if (vals) vals_out[zeros] = vals[i];
            ++zeros;
        }
    }
    size_t ones = zeros;
    for (size_t i = 0; i < n; ++i) {
        if (((keys[i] >> b) & 1u) != 0u) {
            keys_out[ones] = keys[i];
            if (vals) vals_out[ones] = vals[i];
            ++ones;
        }
    }
    return zeros;
}

/*
 * LSD radix sort by one-bit stable splits over bits [begin_bit, end_bit),
 * lowest bit first ([CIS 565] radix sort built on scan).  With the full
 * range [0, 32) the result is the keys in ascending order, ties in input
 * order.  vals_in / vals_out may both be NULL (keys only).  The result
 * always lands in keys_out / vals_out; an empty bit range copies.
 * Returns 0, or -1 on bad arguments or if scratch cannot be allocated.
 */
int orc_split_radix(const uint32_t *keys_in, const uint32_t *vals_in,
                    uint32_t *keys_out, uint32_t *vals_out, size_t n,
                    int begin_bit, int end_bit)
{
    if (begin_bit < 0 || end_bit > 32 || begin_bit > end_bit) return -1;
    if ((vals_in == NULL) != (vals_out == NULL)) return -1;
    if (n == 0) return 0;
    uint32_t *ka = (uint32_t *)malloc(n * sizeof(uint32_t));
    uint32_t *va = vals_in ? (uint32_t *)malloc(n * sizeof(uint32_t)) : NULL;
    uint32_t *kb = (uint32_t *)malloc(n * sizeof(uint32_t));
    uint32_t *vb = vals_in ? (uint32_t *)malloc(n * sizeof(uint32_t)) : NULL;
    if (!ka || !kb || (vals_in && (!va || !vb))) {
        free(ka); free(va); free(kb); free(vb);
        return -1;
    }
    memcpy(ka, keys_in, n * sizeof(uint32_t));
    if (vals_in) memcpy(va, vals_in, n * sizeof(uint32_t));
    for (int b = begin_bit; b < end_bit; ++b) {
        split_by_bit(ka, va, kb, vb, n, b);
        uint32_t *t = ka; ka = kb; kb = t;
        t = va; va = vb; vb = t;
    }
    memcpy(keys_out, ka, n * sizeof(uint32_t));
    if (vals_in) memcpy(vals_out, va, n * sizeof(uint32_t));
    free(ka); free(va); free(kb); free(vb);
    return 0;
}

/*
 * Parameterised predicates ("The CUDA Handbook, ch. 13: Stream compaction":
 * the single-pass compaction "is easily modified to evaluate more-complicated
 * predicates").  Either a comparison of the element with an operand in the
 * dtype's own order -- int32 signed, uint32 unsigned, float32 IEEE 754, where
 * every comparison with NaN is false except "not equal" -- or a test of the
 * raw bits under a mask.  value holds the operand's 32-bit pattern.
 */
enum { ORC_LT = 0, ORC_LE = 1, ORC_GT = 2, ORC_GE = 3, ORC_EQ = 4, ORC_NE = 5,
       ORC_MASK_EQ = 6, ORC_MASK_NE = 7 };

static int keep_cmp(uint32_t bits, int dtype, int cmp, uint32_t value, uint32_t mask)
{
    if (cmp == ORC_MASK_EQ) return (bits & mask) == value;
    if (cmp == ORC_MASK_NE) return (bits & mask) != value;
    if (dtype == ORC_F32) {
        const float x = bits_to_float(bits), v = bits_to_float(value);
        switch (cmp) {
        case ORC_LT: return x < v;
        case ORC_LE: return x <= v;
        case ORC_GT: return x > v;
        case ORC_GE: return x >= v;
        case ORC_EQ: return x == v;
        default: return x != v;
        }
    }
    if (dtype == ORC_I32) {
        int32_t x, v;
        memcpy(&x, &bits, sizeof x);
        memcpy(&v, &value, sizeof v);
        switch (cmp) {
        case ORC_LT: return x < v;
        case ORC_LE: return x <= v;
        case ORC_GT: return x > v;
        case ORC_GE: return x >= v;
        case ORC_EQ: return x == v;
        default: return x != v;
        }
    }
    switch (cmp) {
    case ORC_LT: return bits < value;
    case ORC_LE: return bits <= value;
    case ORC_GT: return bits > value;
    case ORC_GE: return bits >= value;
    case ORC_EQ: return bits == value;
    default: return bits != value;
    }
}

/* Stable select-if with a parameterised predicate; returns the kept count. */
size_t orc_select_if_cmp(const uint32_t *in, uint32_t *out, size_t n, int dtype, int cmp,
                         uint32_t value, uint32_t mask)
{
    size_t m = 0;
    for (size_t i = 0; i < n; ++i) {
        if (keep_cmp(in[i], dtype, cmp, value, mask)) {
            out[m] = in[i];
            ++m;
        }
    }
    return m;
}

/* Stable partition with a parameterised predicate, kept half first. */
size_t orc_partition_cmp(const uint32_t *in, uint32_t *out, size_t n, int dtype, int cmp,
                         uint32_t value, uint32_t mask)
{
    size_t first = 0;
    for (size_t i = 0; i < n; ++i) {
        if (keep_cmp(in[i], dtype, cmp, value, mask)) {
            out[first] = in[i];
            ++first;
        }
    }
    size_t second = first;
    for (size_t i = 0; i < n; ++i) {
        if (!keep_cmp(in[i], dtype, cmp, value, mask)) {
            out[second] = in[i];
            ++second;
        }
    }
    return first;
}

/*
 * Full-width LSD radix sort in the key dtype's order: int32 signed, uint32,
 * float32 in IEEE 754 totalOrder (-NaN < -inf < ... < -0 < +0 < ... < +inf <
 * +NaN).  Each key is mapped to an unsigned key that ascends in that order
 * (int32: flip the sign bit; float32: flip the sign bit of a positive
 * pattern, every bit of a negative one), sorted by the one-bit splits of
 * orc_split_radix over bits [0, 32), and mapped back.  Stable; vals may be
 * NULL.  Returns 0, or -1 on bad arguments or allocation failure.
 */
static uint32_t to_order_key(uint32_t bits, int dtype)
{
    if (dtype == ORC_I32) return bits ^ 0x80000000u;
    if (dtype == ORC_F32) return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    return bits;
}

static uint32_t from_order_key(uint32_t key, int dtype)
{
    if (dtype == ORC_I32) return key ^ 0x80000000u;
    if (dtype == ORC_F32) return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
    return key;
}

int orc_radix_sort(const uint32_t *keys_in, const uint32_t *vals_in, uint32_t *keys_out,
                   uint32_t *vals_out, size_t n, int dtype)
{
    if (dtype != ORC_I32 && dtype != ORC_U32 && dtype != ORC_F32) return -1;
    if (n == 0) return 0;
    uint32_t *k = (uint32_t *)malloc(n * sizeof(uint32_t));
    if (!k) return -1;
    for (size_t i = 0; i < n; ++i) k[i] = to_order_key(keys_in[i], dtype);
    const int rc = orc_split_radix(k, vals_in, keys_out, vals_out, n, 0, 32);
    free(k);
    if (rc != 0) return rc;
    for (size_t i = 0; i < n; ++i) keys_out[i] = from_order_key(keys_out[i], dtype);
    return 0;
}

/*
 * How many positions of an unordered result differ from the stable one.
 * Reported beside the atomic-counter comparator, never used as a pass/fail
 * gate ([Day 33] countOutOfOrder).
 */
size_t orc_count_out_of_order(const uint32_t *got, const uint32_t *want,
                              size_t m)
{
    size_t differ = 0;
    for (size_t k = 0; k < m; ++k) differ += (size_t)(got[k] != want[k]);
    return differ;
}
