// api.cu -- the C ABI of libgc (include/gc.h): argument checks on the host,
// workspace sizing, and dispatch to the launchers.  Nothing here touches the
// GPU before every argument has been checked, so argument errors are
// reported without any CUDA call.
#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/gc.h"
#include "../../include/gc_testing.h"
#include "gc_internal.h"

namespace gch {

cudaError_t reset_tiles(uint8_t *ws, size_t tiles, cudaStream_t s, bool skip_first_tile)
{
    // [kTileCtrOff, kHeaderBytes) holds only the tile counter (and padding).
    cudaError_t e = cudaMemsetAsync(ws + kTileCtrOff, 0,
                                    (kHeaderBytes - kTileCtrOff) + status_bytes(tiles), s);
    if (e == cudaSuccess && skip_first_tile) e = cudaMemsetAsync(ws + kTileCtrOff, 1, 1, s);
    return e;
}

cudaError_t clear_accumulators(uint8_t *ws, cudaStream_t s)
{
    // [0, 8) is the error word and its tile, [kHdrBarArrive, kHeaderBytes)
    // the start barrier's counter and the tile counter; the rest of the
    // header is scratch (the barrier's epoch among it: any value will do).
    return cudaMemsetAsync(ws + 8, 0, kHdrBarArrive - 8, s);
}

static std::atomic<bool> g_force_fallback{false};

bool force_fallback() { return g_force_fallback.load(std::memory_order_relaxed); }

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

int persistent_grid(const void *kernel, int threads, size_t smem, uint32_t tiles)
{
    // A kernel's shared-memory attribute and occupancy do not change while the
    // process runs: set and query them once per (kernel, device, shape).
    struct Entry {
        const void *kernel;
        int dev, threads;
        size_t smem;
        int per_sm;
    };
    static std::mutex mu;
    static Entry cache[128];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry &c = cache[i];
            if (c.kernel == kernel && c.dev == dev && c.threads == threads && c.smem == smem) {
                per_sm = c.per_sm;
                break;
            }
        }
    }
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess)
            return -1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
                cudaSuccess ||
            per_sm <= 0)
            return -1;
        std::lock_guard<std::mutex> lock(mu);
        if (used < 128) cache[used++] = Entry{kernel, dev, threads, smem, per_sm};
    }
    const long long grid = (long long)per_sm * sm_count();
    return int(grid < (long long)tiles ? grid : (long long)tiles);
}

}  // namespace gch

namespace {

using namespace gch;

bool valid_dtype(int dt) { return dt == GC_I32 || dt == GC_U32 || dt == GC_F32; }
bool valid_pred(int p) { return p == GC_PRED_NONZERO || p == GC_PRED_ODD || p == GC_PRED_EVEN; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool overlap(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

gc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GC_OK : GC_ERR_CUDA; }

// Checks shared by every element-wise entry point.
gc_status check_common(const void *in, const void *out, size_t n, void *ws, size_t ws_bytes,
                       gc_op op, gc_dtype dt)
{
    if (n > GC_MAX_ELEMENTS) return GC_ERR_INVALID_VALUE;
    if (!valid_dtype(dt)) return GC_ERR_INVALID_VALUE;
    if (ws == nullptr) return GC_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GC_ERR_MISALIGNED;
    if (ws_bytes < gc_workspace_bytes(op, n, dt)) return GC_ERR_WORKSPACE_TOO_SMALL;
    if (n > 0) {
        if (in == nullptr || out == nullptr) return GC_ERR_INVALID_VALUE;
        if (!aligned4(in) || !aligned4(out)) return GC_ERR_MISALIGNED;
        if (overlap(ws, ws_bytes, in, 4 * n) || overlap(ws, ws_bytes, out, 4 * n))
            return GC_ERR_INVALID_VALUE;
    }
    return GC_OK;
}

gc_status check_select_like(const void *in, const void *out, const uint32_t *count, size_t n,
                            gc_dtype dt, gc_pred p, void *ws, size_t ws_bytes, gc_op op)
{
    gc_status st = check_common(in, out, n, ws, ws_bytes, op, dt);
    if (st != GC_OK) return st;
    if (!valid_pred(p)) return GC_ERR_INVALID_VALUE;
    if (dt == GC_F32 && p != GC_PRED_NONZERO) return GC_ERR_UNSUPPORTED;
    if (count == nullptr) return GC_ERR_INVALID_VALUE;
    if (!aligned4(count)) return GC_ERR_MISALIGNED;
    if (n > 0 && overlap(in, 4 * n, out, 4 * n)) return GC_ERR_INVALID_VALUE;
    if (overlap(count, 4, out, 4 * n) || overlap(count, 4, in, 4 * n) ||
        overlap(count, 4, ws, ws_bytes))
        return GC_ERR_INVALID_VALUE;
    return GC_OK;
}

// Pairing, alignment and aliasing rules of the radix entry points: keys and
// payloads come both or keys alone, each input may equal its output, and no
// other pair of the four arrays (or the workspace) overlaps.
gc_status check_radix_arrays(const void *keys_in, const uint32_t *vals_in, const void *keys_out,
                             const uint32_t *vals_out, size_t n, void *ws, size_t ws_bytes)
{
    if ((vals_in == nullptr) != (vals_out == nullptr)) return GC_ERR_INVALID_VALUE;
    if (n == 0) return GC_OK;
    const size_t b = 4 * n;
    if (keys_in != keys_out && overlap(keys_in, b, keys_out, b)) return GC_ERR_INVALID_VALUE;
    if (vals_in != nullptr) {
        if (!aligned4(vals_in) || !aligned4(vals_out)) return GC_ERR_MISALIGNED;
        if (vals_in != vals_out && overlap(vals_in, b, vals_out, b)) return GC_ERR_INVALID_VALUE;
        const void *keys[2] = {keys_in, keys_out};
        const void *vals[2] = {vals_in, vals_out};
        for (const void *k : keys)
            for (const void *v : vals)
                if (overlap(k, b, v, b)) return GC_ERR_INVALID_VALUE;
        if (overlap(ws, ws_bytes, vals_in, b) || overlap(ws, ws_bytes, vals_out, b))
            return GC_ERR_INVALID_VALUE;
    }
    return GC_OK;
}

// Which select-if: the stable one, or the atomic comparison path with one
// atomic per survivor or per tile.
enum class SelectKind { Stable, AtomicElem, AtomicTile };

gc_status select_like(SelectKind kind, const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                      gc_dtype dt, gc_pred p, void *d_ws, size_t ws_bytes, cudaStream_t s,
                      const LaunchOpts &o)
{
    const bool atomic = kind != SelectKind::Stable;
    const gc_op op = atomic ? GC_OP_SELECT_IF_ATOMIC : GC_OP_SELECT_IF;
    gc_status st = check_select_like(d_in, d_out, d_count, n, dt, p, d_ws, ws_bytes, op);
    if (st != GC_OK) return st;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count, 0, sizeof(uint32_t), s));
    if (atomic)
        return from_cuda(launch_select_atomic(d_in, d_out, d_count, uint32_t(n), dt, p, s,
                                              kind == SelectKind::AtomicTile));
    return from_cuda(launch_select(d_in, d_out, d_count, uint32_t(n), dt, p,
                                   static_cast<uint8_t *>(d_ws), s, o));
}

}  // namespace

extern "C" {

const char *gc_status_string(gc_status status)
{
    switch (status) {
    case GC_OK: return "GC_OK";
    case GC_ERR_INVALID_VALUE: return "GC_ERR_INVALID_VALUE: bad argument";
    case GC_ERR_UNSUPPORTED: return "GC_ERR_UNSUPPORTED: predicate not defined for this dtype";
    case GC_ERR_WORKSPACE_TOO_SMALL: return "GC_ERR_WORKSPACE_TOO_SMALL";
    case GC_ERR_MISALIGNED: return "GC_ERR_MISALIGNED: pointer alignment";
    case GC_ERR_CUDA: return "GC_ERR_CUDA: CUDA call or launch failed";
    case GC_ERR_TIMEOUT: return "GC_ERR_TIMEOUT: a look-back wait gave up on the device";
    case GC_ERR_DEVICE_CHECK: return "GC_ERR_DEVICE_CHECK: a kernel refused an out-of-range store";
    }
    return "unknown gc_status";
}

const char *gc_version(void) { return "libgc 0.1 (sm_103a)"; }

size_t gc_workspace_bytes(gc_op op, size_t n, gc_dtype dtype)
{
    if (n > GC_MAX_ELEMENTS) return 0;
    const size_t status = status_bytes(max_tiles(n));
    switch (op) {
    case GC_OP_EXCLUSIVE_SCAN:
    case GC_OP_INCLUSIVE_SCAN:
        if (!valid_dtype(dtype)) return 0;
        return kHeaderBytes + status + (dtype == GC_F32 ? status : 0);
    case GC_OP_SELECT_IF:
    case GC_OP_PARTITION:
    case GC_OP_SELECT_IF_ATOMIC:
        if (!valid_dtype(dtype)) return 0;
        return kHeaderBytes + status;
    case GC_OP_RADIX_SORT:
        if (!valid_dtype(dtype)) return 0;
        return digit_table_offset(n) + digit_table_bytes(n);
    case GC_OP_REDUCE:
    case GC_OP_COUNT_IF:
        if (!valid_dtype(dtype)) return 0;
        return kHeaderBytes + status;
    case GC_OP_SPLIT_RADIX:
        return radix_temp_offset(n) + 2 * radix_temp_stride(n);
    }
    return 0;
}

size_t gc_tile_elements(gc_op op)
{
    switch (op) {
    case GC_OP_EXCLUSIVE_SCAN:
    case GC_OP_INCLUSIVE_SCAN: return scan_tile_elems();
    case GC_OP_SELECT_IF: return select_tile_elems();
    case GC_OP_PARTITION: return partition_tile_elems();
    case GC_OP_SPLIT_RADIX: return split_tile_elems();
    case GC_OP_RADIX_SORT: return kDigitTile;
    case GC_OP_SELECT_IF_ATOMIC: return atomic_tile_elems();
    case GC_OP_REDUCE:
    case GC_OP_COUNT_IF: return 4 * kReduceThreads;
    }
    return 0;
}

gc_status gc_workspace_init(void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    if (d_ws == nullptr) return GC_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0) return GC_ERR_MISALIGNED;
    return from_cuda(cudaMemsetAsync(d_ws, 0, ws_bytes, stream));
}

static gc_status scan_entry(const void *d_in, void *d_out, void *d_total, size_t n,
                            gc_dtype dtype, void *d_ws, size_t ws_bytes, cudaStream_t stream,
                            bool inclusive, const LaunchOpts &o = LaunchOpts{})
{
    gc_status st = check_common(d_in, d_out, n, d_ws, ws_bytes, GC_OP_EXCLUSIVE_SCAN, dtype);
    if (st != GC_OK) return st;
    if (n > 0 && d_in != d_out && overlap(d_in, 4 * n, d_out, 4 * n)) return GC_ERR_INVALID_VALUE;
    if (d_total != nullptr) {
        if (!aligned4(d_total)) return GC_ERR_MISALIGNED;
        if (overlap(d_total, 4, d_out, 4 * n) || overlap(d_total, 4, d_in, 4 * n) ||
            overlap(d_total, 4, d_ws, ws_bytes))
            return GC_ERR_INVALID_VALUE;
    }
    if (n == 0)
        return d_total ? from_cuda(cudaMemsetAsync(d_total, 0, 4, stream)) : GC_OK;
    return from_cuda(launch_scan(d_in, d_out, d_total, uint32_t(n), dtype,
                                 static_cast<uint8_t *>(d_ws), stream, o, inclusive));
}

gc_status gc_exclusive_scan(const void *d_in, void *d_out, void *d_total, size_t n,
                            gc_dtype dtype, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    return scan_entry(d_in, d_out, d_total, n, dtype, d_ws, ws_bytes, stream, false);
}

gc_status gc_inclusive_scan(const void *d_in, void *d_out, void *d_total, size_t n,
                            gc_dtype dtype, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    return scan_entry(d_in, d_out, d_total, n, dtype, d_ws, ws_bytes, stream, true);
}

gc_status gc_select_if(const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                       gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                       cudaStream_t stream)
{
    return select_like(SelectKind::Stable, d_in, d_out, d_count, n, dtype, pred, d_ws, ws_bytes,
                       stream, LaunchOpts{});
}

gc_status gc_select_if_atomic(const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                              gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                              cudaStream_t stream)
{
    return select_like(SelectKind::AtomicElem, d_in, d_out, d_count, n, dtype, pred, d_ws,
                       ws_bytes, stream, LaunchOpts{});
}

gc_status gc_select_if_atomic_tile(const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                                   gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                                   cudaStream_t stream)
{
    return select_like(SelectKind::AtomicTile, d_in, d_out, d_count, n, dtype, pred, d_ws,
                       ws_bytes, stream, LaunchOpts{});
}

gc_status gc_partition(const void *d_in, void *d_out, uint32_t *d_count_true, size_t n,
                       gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                       cudaStream_t stream)
{
    gc_status st = check_select_like(d_in, d_out, d_count_true, n, dtype, pred, d_ws, ws_bytes,
                                     GC_OP_PARTITION);
    if (st != GC_OK) return st;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count_true, 0, sizeof(uint32_t), stream));
    return from_cuda(launch_partition(d_in, d_out, d_count_true, uint32_t(n), dtype, pred,
                                      static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}));
}

// Order-preserving unsigned key of a 32-bit pattern in the dtype's order
// (the device applies the same map to every element).
static uint32_t order_key(uint32_t bits, gc_dtype dt)
{
    if (dt == GC_I32) return bits ^ 0x80000000u;
    if (dt == GC_F32) return bits ^ ((bits >> 31) ? 0xFFFFFFFFu : 0x80000000u);
    return bits;
}

// Keep-interval of a comparison, in keys: [lo, hi], or nothing / everything.
static void keep_interval(gc_cmp cmp, uint32_t operand, gc_dtype dt, CmpSpec &c)
{
    // signed 64-bit: low - 1 below key 0 and high + 1 above 2^32 - 1 stay empty
    auto set = [&](int64_t lo, int64_t hi, bool inv) {
        if (lo > hi) {  // empty interval: keep nothing (the complement of everything)
            c.lo = 0u;
            c.span = 0xFFFFFFFFu;
            c.invert = inv ? 0u : 1u;
        } else {
            c.lo = uint32_t(lo);
            c.span = uint32_t(hi - lo);
            c.invert = inv ? 1u : 0u;
        }
    };
    int64_t kmin = 0, kmax = 0xFFFFFFFFll, low, high;
    if (dt == GC_F32) {
        const bool nan = (operand & 0x7F800000u) == 0x7F800000u && (operand & 0x007FFFFFu) != 0u;
        if (nan) {  // every comparison with NaN is false, except "not equal"
            set(1, 0, cmp == GC_CMP_NE);
            return;
        }
        kmin = order_key(0xFF800000u, dt);  // -inf
        kmax = order_key(0x7F800000u, dt);  // +inf
        const bool zero = (operand & 0x7FFFFFFFu) == 0u;
        low = zero ? order_key(0x80000000u, dt) : order_key(operand, dt);   // -0.0 first
        high = zero ? order_key(0x00000000u, dt) : order_key(operand, dt);  // +0.0 last
    } else {
        low = high = order_key(operand, dt);
    }
    switch (cmp) {
    case GC_CMP_LT: set(kmin, low - 1, false); break;  // low == kmin gives an empty interval
    case GC_CMP_LE: set(kmin, high, false); break;
    case GC_CMP_GT: set(high + 1, kmax, false); break;
    case GC_CMP_GE: set(low, kmax, false); break;
    case GC_CMP_EQ: set(low, high, false); break;
    default: set(low, high, true); break;  // GC_CMP_NE
    }
}

static bool cmp_spec(const gc_predicate *pred, gc_dtype dt, CmpSpec &c)
{
    if (pred == nullptr) return false;
    const int cmp = int(pred->cmp);
    if (cmp < GC_CMP_LT || cmp > GC_CMP_MASK_NE) return false;
    c = CmpSpec{};
    if (cmp >= GC_CMP_MASK_EQ) {
        c.is_mask = 1u;
        c.mask = pred->mask;
        c.value = pred->operand;
        c.invert = cmp == GC_CMP_MASK_NE ? 1u : 0u;
    } else {
        keep_interval(gc_cmp(cmp), pred->operand, dt, c);
    }
    return true;
}

gc_status gc_select_if_pred(const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                            gc_dtype dtype, const gc_predicate *pred, void *d_ws, size_t ws_bytes,
                            cudaStream_t stream)
{
    CmpSpec c;
    if (!cmp_spec(pred, dtype, c)) return GC_ERR_INVALID_VALUE;
    gc_status st = check_select_like(d_in, d_out, d_count, n, dtype, GC_PRED_NONZERO, d_ws,
                                     ws_bytes, GC_OP_SELECT_IF);
    if (st != GC_OK) return st;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count, 0, sizeof(uint32_t), stream));
    return from_cuda(launch_select_cmp(d_in, d_out, d_count, uint32_t(n), dtype, c,
                                       static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}));
}

gc_status gc_partition_pred(const void *d_in, void *d_out, uint32_t *d_count_true, size_t n,
                            gc_dtype dtype, const gc_predicate *pred, void *d_ws, size_t ws_bytes,
                            cudaStream_t stream)
{
    CmpSpec c;
    if (!cmp_spec(pred, dtype, c)) return GC_ERR_INVALID_VALUE;
    gc_status st = check_select_like(d_in, d_out, d_count_true, n, dtype, GC_PRED_NONZERO, d_ws,
                                     ws_bytes, GC_OP_PARTITION);
    if (st != GC_OK) return st;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count_true, 0, sizeof(uint32_t), stream));
    return from_cuda(launch_partition_cmp(d_in, d_out, d_count_true, uint32_t(n), dtype, c,
                                          static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}));
}

gc_status gc_split_radix(const uint32_t *d_keys_in, const uint32_t *d_vals_in,
                         uint32_t *d_keys_out, uint32_t *d_vals_out, size_t n, int begin_bit,
                         int end_bit, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    gc_status st = check_common(d_keys_in, d_keys_out, n, d_ws, ws_bytes, GC_OP_SPLIT_RADIX, GC_U32);
    if (st != GC_OK) return st;
    if (begin_bit < 0 || end_bit > 32 || begin_bit > end_bit) return GC_ERR_INVALID_VALUE;
    if ((st = check_radix_arrays(d_keys_in, d_vals_in, d_keys_out, d_vals_out, n, d_ws, ws_bytes)) != GC_OK)
        return st;
    if (n == 0) return GC_OK;
    return from_cuda(launch_split_radix(d_keys_in, d_vals_in, d_keys_out, d_vals_out, uint32_t(n),
                                        begin_bit, end_bit, static_cast<uint8_t *>(d_ws), stream,
                                        LaunchOpts{}));
}

gc_status gc_radix_sort(const void *d_keys_in, const uint32_t *d_vals_in, void *d_keys_out,
                        uint32_t *d_vals_out, size_t n, gc_dtype dtype, void *d_ws, size_t ws_bytes,
                        cudaStream_t stream)
{
    gc_status st = check_common(d_keys_in, d_keys_out, n, d_ws, ws_bytes, GC_OP_RADIX_SORT, dtype);
    if (st != GC_OK) return st;
    if ((st = check_radix_arrays(d_keys_in, d_vals_in, d_keys_out, d_vals_out, n, d_ws, ws_bytes)) != GC_OK)
        return st;
    if (n == 0) return GC_OK;
    // Order-preserving key x ^ (signfill(x) & neg) ^ flip (PredKeyBitClear).
    const uint32_t neg = dtype == GC_F32 ? 0x7FFFFFFFu : 0u;
    const uint32_t flip = dtype == GC_U32 ? 0u : 0x80000000u;
    return from_cuda(launch_radix_sort_digits(static_cast<const uint32_t *>(d_keys_in), d_vals_in,
                                              static_cast<uint32_t *>(d_keys_out), d_vals_out,
                                              uint32_t(n), neg, flip, static_cast<uint8_t *>(d_ws),
                                              stream, LaunchOpts{}));
}

// ---------------------------------------------------------------- sharded calls

gc_status gc_reduce(const void *d_in, void *d_total, size_t n, gc_dtype dtype, void *d_ws,
                    size_t ws_bytes, cudaStream_t stream)
{
    gc_status st = check_common(d_in, d_in, n, d_ws, ws_bytes, GC_OP_REDUCE, dtype);
    if (st != GC_OK) return st;
    if (d_total == nullptr) return GC_ERR_INVALID_VALUE;
    if (!aligned4(d_total)) return GC_ERR_MISALIGNED;
    if (overlap(d_total, 4, d_in, 4 * n) || overlap(d_total, 4, d_ws, ws_bytes))
        return GC_ERR_INVALID_VALUE;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_total, 0, 4, stream));
    return from_cuda(launch_reduce(d_in, d_total, uint32_t(n), dtype, static_cast<uint8_t *>(d_ws),
                                   stream));
}

gc_status gc_count_if(const void *d_in, uint32_t *d_count, size_t n, gc_dtype dtype, gc_pred pred,
                      void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    gc_status st = check_common(d_in, d_in, n, d_ws, ws_bytes, GC_OP_COUNT_IF, dtype);
    if (st != GC_OK) return st;
    if (!valid_pred(pred)) return GC_ERR_INVALID_VALUE;
    if (dtype == GC_F32 && pred != GC_PRED_NONZERO) return GC_ERR_UNSUPPORTED;
    if (d_count == nullptr) return GC_ERR_INVALID_VALUE;
    if (!aligned4(d_count)) return GC_ERR_MISALIGNED;
    if (overlap(d_count, 4, d_in, 4 * n) || overlap(d_count, 4, d_ws, ws_bytes))
        return GC_ERR_INVALID_VALUE;
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count, 0, 4, stream));
    return from_cuda(launch_count_if(d_in, d_count, uint32_t(n), dtype, pred,
                                     static_cast<uint8_t *>(d_ws), stream));
}

gc_status gc_exclusive_scan_carry(const void *d_in, void *d_out, void *d_total, size_t n,
                                  gc_dtype dtype, const void *d_carry, void *d_ws,
                                  size_t ws_bytes, cudaStream_t stream)
{
    if (d_carry == nullptr) return GC_ERR_INVALID_VALUE;
    if (!aligned4(d_carry)) return GC_ERR_MISALIGNED;
    gc_status st = check_common(d_in, d_out, n, d_ws, ws_bytes, GC_OP_EXCLUSIVE_SCAN, dtype);
    if (st != GC_OK) return st;
    if (n > 0 && d_in != d_out && overlap(d_in, 4 * n, d_out, 4 * n)) return GC_ERR_INVALID_VALUE;
    if (overlap(d_carry, 4, d_out, 4 * n) || overlap(d_carry, 4, d_ws, ws_bytes))
        return GC_ERR_INVALID_VALUE;
    if (d_total != nullptr) {
        if (!aligned4(d_total)) return GC_ERR_MISALIGNED;
        if (overlap(d_total, 4, d_out, 4 * n) || overlap(d_total, 4, d_in, 4 * n) ||
            overlap(d_total, 4, d_ws, ws_bytes) || overlap(d_total, 4, d_carry, 4))
            return GC_ERR_INVALID_VALUE;
    }
    if (n == 0)  // the total of nothing after the carry is the carry
        return d_total ? from_cuda(cudaMemcpyAsync(d_total, d_carry, 4, cudaMemcpyDeviceToDevice,
                                                   stream))
                       : GC_OK;
    return from_cuda(launch_scan(d_in, d_out, d_total, uint32_t(n), dtype,
                                 static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}, false,
                                 d_carry));
}

gc_status gc_select_if_at(const void *d_in, void *d_out, size_t out_capacity,
                          const uint64_t *d_base, uint32_t *d_count, size_t n, gc_dtype dtype,
                          gc_pred pred, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    if (d_base == nullptr) return GC_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(d_base) & 7u) != 0) return GC_ERR_MISALIGNED;
    gc_status st = check_select_like(d_in, d_out, d_count, n, dtype, pred, d_ws, ws_bytes,
                                     GC_OP_SELECT_IF);
    if (st != GC_OK) return st;
    if (n > 0) {
        if (out_capacity == 0 || out_capacity > (size_t(1) << 62)) return GC_ERR_INVALID_VALUE;
        const size_t ob = 4 * out_capacity;
        if (overlap(d_out, ob, d_in, 4 * n) || overlap(d_out, ob, d_ws, ws_bytes) ||
            overlap(d_out, ob, d_count, 4) || overlap(d_out, ob, d_base, 8))
            return GC_ERR_INVALID_VALUE;
    }
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count, 0, sizeof(uint32_t), stream));
    return from_cuda(launch_select(d_in, d_out, d_count, uint32_t(n), dtype, pred,
                                   static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}, d_base,
                                   uint64_t(out_capacity)));
}

gc_status gc_partition_at(const void *d_in, void *d_out, size_t out_capacity,
                          const uint64_t *d_offsets, uint32_t *d_count_true, size_t n,
                          gc_dtype dtype, gc_pred pred, void *d_ws, size_t ws_bytes,
                          cudaStream_t stream)
{
    if (d_offsets == nullptr) return GC_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(d_offsets) & 7u) != 0) return GC_ERR_MISALIGNED;
    gc_status st = check_select_like(d_in, d_out, d_count_true, n, dtype, pred, d_ws, ws_bytes,
                                     GC_OP_PARTITION);
    if (st != GC_OK) return st;
    if (n > 0) {
        if (out_capacity < n || out_capacity > (size_t(1) << 62)) return GC_ERR_INVALID_VALUE;
        const size_t ob = 4 * out_capacity;
        if (overlap(d_out, ob, d_in, 4 * n) || overlap(d_out, ob, d_ws, ws_bytes) ||
            overlap(d_out, ob, d_count_true, 4) || overlap(d_out, ob, d_offsets, 16))
            return GC_ERR_INVALID_VALUE;
    }
    if (n == 0) return from_cuda(cudaMemsetAsync(d_count_true, 0, sizeof(uint32_t), stream));
    return from_cuda(launch_partition_at(d_in, d_out, uint64_t(out_capacity), d_offsets,
                                         d_count_true, uint32_t(n), dtype, pred,
                                         static_cast<uint8_t *>(d_ws), stream, LaunchOpts{}));
}

gc_status gc_shard_offsets(gc_op op, gc_dtype dtype, const uint32_t *d_totals,
                           const uint64_t *h_sizes, size_t parts, size_t rank, void *d_offsets,
                           cudaStream_t stream)
{
    if (op != GC_OP_EXCLUSIVE_SCAN && op != GC_OP_SELECT_IF && op != GC_OP_PARTITION)
        return GC_ERR_INVALID_VALUE;
    if (!valid_dtype(dtype)) return GC_ERR_INVALID_VALUE;
    if (parts == 0 || parts > GC_MAX_SHARDS || rank >= parts) return GC_ERR_INVALID_VALUE;
    if (d_totals == nullptr || d_offsets == nullptr) return GC_ERR_INVALID_VALUE;
    if (!aligned4(d_totals)) return GC_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(d_offsets) & (op == GC_OP_EXCLUSIVE_SCAN ? 3u : 7u)) != 0)
        return GC_ERR_MISALIGNED;
    uint64_t before = 0;
    if (op == GC_OP_PARTITION) {
        if (h_sizes == nullptr) return GC_ERR_INVALID_VALUE;
        for (size_t q = 0; q < parts; ++q)
            if (h_sizes[q] > GC_MAX_ELEMENTS) return GC_ERR_INVALID_VALUE;
        for (size_t q = 0; q < rank; ++q) before += h_sizes[q];
    }
    const size_t out_bytes = op == GC_OP_EXCLUSIVE_SCAN ? 4 : (op == GC_OP_PARTITION ? 16 : 8);
    if (overlap(d_offsets, out_bytes, d_totals, 4 * parts)) return GC_ERR_INVALID_VALUE;
    return from_cuda(launch_shard_offsets(op, dtype, d_totals, uint32_t(parts), uint32_t(rank),
                                          before, d_offsets, stream));
}

gc_status gc_query_device_status(void *d_ws, cudaStream_t stream)
{
    if (d_ws == nullptr) return GC_ERR_INVALID_VALUE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GC_ERR_CUDA;
    uint32_t err = 0;
    if (cudaMemcpy(&err, d_ws, sizeof err, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GC_ERR_CUDA;
    if (err != 0) {
        // The error word and its tile, and the start barrier's counter (a
        // wait that ran out leaves it marked so that no later barrier can
        // complete early).
        const uint32_t zero[2] = {0, 0};
        uint8_t *ws = static_cast<uint8_t *>(d_ws);
        if (cudaMemcpy(ws, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(ws + kHdrBarArrive, zero, sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess)
            return GC_ERR_CUDA;
        return (err == GC_ERR_TIMEOUT || err == GC_ERR_DEVICE_CHECK) ? gc_status(err) : GC_ERR_CUDA;
    }
    return GC_OK;
}

gc_status gc_testing_select_if_skip_tile0(const void *d_in, void *d_out, uint32_t *d_count,
                                          size_t n, gc_dtype dtype, gc_pred pred, void *d_ws,
                                          size_t ws_bytes, uint64_t timeout_ns,
                                          cudaStream_t stream)
{
    if (n <= gch::select_tile_elems()) return GC_ERR_INVALID_VALUE;
    LaunchOpts o;
    o.timeout_ns = timeout_ns;
    o.skip_first_tile = true;
    return select_like(SelectKind::Stable, d_in, d_out, d_count, n, dtype, pred, d_ws, ws_bytes,
                       stream, o);
}

void gc_testing_force_fallback(int on) { g_force_fallback.store(on != 0); }

gc_status gc_testing_exclusive_scan_stalled_barrier(const void *d_in, void *d_out, void *d_total,
                                                    size_t n, gc_dtype dtype, void *d_ws,
                                                    size_t ws_bytes, uint64_t timeout_ns,
                                                    cudaStream_t stream)
{
    gc_status st = check_common(d_in, d_out, n, d_ws, ws_bytes, GC_OP_EXCLUSIVE_SCAN, dtype);
    if (st != GC_OK) return st;
    if (n == 0 || !aligned16(d_in)) return GC_ERR_INVALID_VALUE;
    // The top byte of the little-endian arrival counter: the mark a barrier
    // wait that ran out leaves.
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    if (cudaMemsetAsync(ws + kHdrBarArrive + 3, 0x80, 1, stream) != cudaSuccess) return GC_ERR_CUDA;
    LaunchOpts o;
    o.timeout_ns = timeout_ns;
    return scan_entry(d_in, d_out, d_total, n, dtype, d_ws, ws_bytes, stream, false, o);
}

}  // extern "C"
