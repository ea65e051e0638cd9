// noalloc.cu -- gc_select_if_noalloc: stable select-if for callers that
// cannot provide a workspace.
//
// Some callers cannot allocate device memory at the point where they need a
// compaction: a plugin whose host framework owns the whole device memory
// budget and forbids allocations behind its back, or a latency-critical loop
// that must not pay cudaMalloc / cudaFree, which may synchronise the device.
// This entry point needs no workspace argument.  Its scratch (the tile
// counter, the per-tile status words and the header the kernels use) is one
// file-scope device array, kNoallocScratchBytes long, which every GPU that
// loads this library holds until the process exits.
//
// Host code cannot hand the array's name to a kernel: on the host that name
// is a stand-in, not a device address.  So the first call on each device,
// with that device current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and caches it; later calls on that device reuse it.
// Make the first call on a device before any stream capture begins.
//
// Every call shares the one array.  Each call clears the parts that must
// start at zero on its own stream: the persistent kernel its status words,
// inside the kernel; the one-tile-per-CTA fallback the tile counter and its
// status words, with an async memset first.  Calls whose work can overlap on
// the GPU (different streams with no ordering between them) race on the
// array and must not be issued.  The array starts zero-filled, as a
// workspace must.  Failures inside a kernel are recorded in the array's
// error word, which gc_select_if_noalloc_status reads and clears.
//
// The cached address belongs to the device's primary context: a
// cudaDeviceReset destroys that context, and with it the array and every
// cached value of this library, so the library must not be used across a
// device reset.
#include <cstring>
#include <mutex>

#include "../../include/gc.h"
#include "../../include/gc_testing.h"
#include "gc_internal.h"

namespace {

// Header + one status word per 2048 elements for GC_NOALLOC_MAX_ELEMENTS,
// rounded up to a whole KiB: the select-if workspace rule of
// gc_workspace_bytes for 2^28 elements.
constexpr size_t kNoallocScratchBytes = 1049600;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up on the
// first call per device).  Returns nullptr if the runtime refused.
void *scratch_for_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

// The entry point and its test hook: a hook may set the wait limit and mark
// the start barrier before the call.
gc_status select_if_noalloc(const void *d_in, void *d_out, uint32_t *d_count, size_t n,
                            gc_dtype dtype, gc_pred pred, cudaStream_t stream,
                            const gch::LaunchOpts &o, bool stall_barrier)
{
    if (n > GC_NOALLOC_MAX_ELEMENTS) return GC_ERR_INVALID_VALUE;
    if (dtype != GC_I32 && dtype != GC_U32 && dtype != GC_F32) return GC_ERR_INVALID_VALUE;
    if (pred != GC_PRED_NONZERO && pred != GC_PRED_ODD && pred != GC_PRED_EVEN)
        return GC_ERR_INVALID_VALUE;
    if (dtype == GC_F32 && pred != GC_PRED_NONZERO) return GC_ERR_UNSUPPORTED;
    if (d_count == nullptr) return GC_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(d_count) & 3u) != 0) return GC_ERR_MISALIGNED;
    if (n > 0) {
        if (d_in == nullptr || d_out == nullptr) return GC_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(d_in) & 3u) != 0 ||
            (reinterpret_cast<uintptr_t>(d_out) & 3u) != 0)
            return GC_ERR_MISALIGNED;
        if (overlaps(d_in, 4 * n, d_out, 4 * n) || overlaps(d_count, 4, d_out, 4 * n) ||
            overlaps(d_count, 4, d_in, 4 * n))
            return GC_ERR_INVALID_VALUE;
    }
    void *scratch = scratch_for_current_device();
    if (scratch == nullptr) return GC_ERR_CUDA;
    if (gc_workspace_bytes(GC_OP_SELECT_IF, n, dtype) > kNoallocScratchBytes)
        return GC_ERR_INVALID_VALUE;
    if (n == 0)
        return cudaMemsetAsync(d_count, 0, sizeof(uint32_t), stream) == cudaSuccess ? GC_OK
                                                                                  : GC_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    if (stall_barrier &&
        cudaMemsetAsync(ws + gch::kHdrBarArrive + 3, 0x80, 1, stream) != cudaSuccess)
        return GC_ERR_CUDA;
    const cudaError_t e = gch::launch_select(d_in, d_out, d_count, uint32_t(n), dtype, pred, ws,
                                             stream, o);
    return e == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace

extern "C" gc_status gc_select_if_noalloc(const void *d_in, void *d_out, uint32_t *d_count,
                                          size_t n, gc_dtype dtype, gc_pred pred,
                                          cudaStream_t stream)
{
    return select_if_noalloc(d_in, d_out, d_count, n, dtype, pred, stream, gch::LaunchOpts{},
                             false);
}

// Reads and clears the device-side error word of the array, as
// gc_query_device_status does for a workspace; after an error also resets
// the start barrier's arrival counter, which a barrier wait that gave up
// leaves marked.  Synchronous: waits for the stream first.
extern "C" gc_status gc_select_if_noalloc_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GC_ERR_CUDA;
    void *scratch = scratch_for_current_device();
    if (scratch == nullptr) return GC_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    uint32_t err = 0;
    if (cudaMemcpy(&err, ws, sizeof err, cudaMemcpyDeviceToHost) != cudaSuccess) return GC_ERR_CUDA;
    if (err == 0) return GC_OK;
    const uint32_t zero[2] = {0, 0};
    if (cudaMemcpy(ws, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(ws + gch::kHdrBarArrive, zero, sizeof(uint32_t), cudaMemcpyHostToDevice) !=
            cudaSuccess)
        return GC_ERR_CUDA;
    return (err == GC_ERR_TIMEOUT || err == GC_ERR_DEVICE_CHECK) ? gc_status(err) : GC_ERR_CUDA;
}

extern "C" gc_status gc_testing_select_if_noalloc_stalled_barrier(const void *d_in, void *d_out,
                                                                   uint32_t *d_count, size_t n,
                                                                   gc_dtype dtype, gc_pred pred,
                                                                   uint64_t timeout_ns,
                                                                   cudaStream_t stream)
{
    // the persistent kernel's path: the one with the start barrier
    if (n == 0 || (reinterpret_cast<uintptr_t>(d_in) & 15u) != 0) return GC_ERR_INVALID_VALUE;
    gch::LaunchOpts o;
    o.timeout_ns = timeout_ns;
    return select_if_noalloc(d_in, d_out, d_count, n, dtype, pred, stream, o, true);
}
