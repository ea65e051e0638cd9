// gc_internal.h -- host-side plumbing shared by the libgc translation units:
// tile configurations, workspace layout arithmetic and the launchers that
// api.cu dispatches to.  Not part of the public ABI (include/gc.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/gc.h"

namespace gch {

// Tile shapes: THREADS threads per CTA, ROWS 16-byte vectors per thread, so
// a tile holds THREADS * 4 * ROWS elements.  Overridable at build time
// (-DGC_SCAN_ROWS=8 ...) for tuning sweeps.
#ifndef GC_SCAN_THREADS
#define GC_SCAN_THREADS 256
#endif
#ifndef GC_SCAN_ROWS
#define GC_SCAN_ROWS 4
#endif
#ifndef GC_SELECT_THREADS
#define GC_SELECT_THREADS 256
#endif
#ifndef GC_SELECT_ROWS
#define GC_SELECT_ROWS 4
#endif
#ifndef GC_PART_THREADS
#define GC_PART_THREADS 256
#endif
#ifndef GC_PART_ROWS
#define GC_PART_ROWS 4
#endif
#ifndef GC_SPLIT_THREADS
#define GC_SPLIT_THREADS 256
#endif
#ifndef GC_SPLIT_ROWS
#define GC_SPLIT_ROWS 4
#endif
// 1: every thread of the CTA takes part in the look-back (THREADS tiles per
// window); 0: warp 0 alone (32 tiles per window).
#ifndef GC_CTA_LOOKBACK
#define GC_CTA_LOOKBACK 0
#endif
// Persistent pipelined kernels: tile shape and the number of tiles in flight
// per CTA (each stage is one tile buffer in shared memory).
#ifndef GC_SCAN_PIPE_THREADS
#define GC_SCAN_PIPE_THREADS 256
#endif
#ifndef GC_SCAN_PIPE_ROWS
#define GC_SCAN_PIPE_ROWS 8
#endif
#ifndef GC_SCAN_PIPE_STAGES
#define GC_SCAN_PIPE_STAGES 3
#endif
constexpr int kScanPipeThreads = GC_SCAN_PIPE_THREADS, kScanPipeRows = GC_SCAN_PIPE_ROWS;
constexpr int kScanPipeStages = GC_SCAN_PIPE_STAGES;
#ifndef GC_SELECT_PIPE_THREADS
#define GC_SELECT_PIPE_THREADS 256
#endif
#ifndef GC_SELECT_PIPE_ROWS
#define GC_SELECT_PIPE_ROWS 8
#endif
#ifndef GC_SELECT_PIPE_STAGES
#define GC_SELECT_PIPE_STAGES 3
#endif
#ifndef GC_PART_PIPE_THREADS
#define GC_PART_PIPE_THREADS 256
#endif
#ifndef GC_PART_PIPE_ROWS
#define GC_PART_PIPE_ROWS 8
#endif
#ifndef GC_PART_PIPE_STAGES
#define GC_PART_PIPE_STAGES 3
#endif
#ifndef GC_SPLIT_PIPE_THREADS
#define GC_SPLIT_PIPE_THREADS 256
#endif
#ifndef GC_SPLIT_PIPE_ROWS
#define GC_SPLIT_PIPE_ROWS 4
#endif
#ifndef GC_SPLIT_PIPE_STAGES
#define GC_SPLIT_PIPE_STAGES 3
#endif
constexpr int kSelectPipeThreads = GC_SELECT_PIPE_THREADS, kSelectPipeRows = GC_SELECT_PIPE_ROWS;
constexpr int kSelectPipeStages = GC_SELECT_PIPE_STAGES;
constexpr int kPartPipeThreads = GC_PART_PIPE_THREADS, kPartPipeRows = GC_PART_PIPE_ROWS;
constexpr int kPartPipeStages = GC_PART_PIPE_STAGES;
constexpr int kSplitPipeThreads = GC_SPLIT_PIPE_THREADS, kSplitPipeRows = GC_SPLIT_PIPE_ROWS;
constexpr int kSplitPipeStages = GC_SPLIT_PIPE_STAGES;
// Minimum resident CTAs per SM the persistent kernels are compiled for
// (the second __launch_bounds__ argument); 0 leaves it out, which lets ptxas
// pick its own register budget for the block size.
#ifndef GC_PIPE_MIN_BLOCKS
#define GC_PIPE_MIN_BLOCKS 0
#endif
constexpr int kPipeMinBlocks = GC_PIPE_MIN_BLOCKS;


constexpr int kScanThreads = GC_SCAN_THREADS, kScanRows = GC_SCAN_ROWS;
constexpr int kSelectThreads = GC_SELECT_THREADS, kSelectRows = GC_SELECT_ROWS;
constexpr int kPartThreads = GC_PART_THREADS, kPartRows = GC_PART_ROWS;
constexpr int kSplitThreads = GC_SPLIT_THREADS, kSplitRows = GC_SPLIT_ROWS;
constexpr int kAtomicThreads = 256, kAtomicRows = 4;
constexpr int kReduceThreads = 256;
constexpr bool kCtaLookback = GC_CTA_LOOKBACK != 0;

constexpr uint32_t tile_elems(int threads, int rows) { return uint32_t(threads) * 4u * uint32_t(rows); }

// Workspaces are sized for the smallest tile any kernel may use, so a
// workspace stays valid whatever tile shape a build picks.
constexpr uint32_t kMinTileElems = 2048;
constexpr size_t kHeaderBytes = 512;
constexpr size_t kHdrBarArrive = 496;  // u32: the persistent kernels' start-barrier counter
constexpr size_t kTileCtrOff = 504;

inline size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t a, size_t b) { return ceil_div(a, b) * b; }

// Bytes of status words a call with `tiles` tiles clears and uses.
inline size_t status_bytes(size_t tiles) { return 8 * tiles; }

// Workspace capacity rules (also what gc_workspace_bytes returns).
inline size_t max_tiles(size_t n) { return ceil_div(n, kMinTileElems) + 1; }
inline size_t radix_temp_offset(size_t n) { return align_up(kHeaderBytes + status_bytes(max_tiles(n)), 256); }
inline size_t radix_temp_stride(size_t n) { return align_up(4 * n, 256); }
// The digit radix sort: keys per tile of its count and scatter kernels, and
// its digit-major count table (256 words per tile) after the ping-pong
// buffers; the scan of that table reports its total in the header.
constexpr uint32_t kDigitTile = 4096;
constexpr uint32_t kHdrDigitScanTotal = 320;
inline size_t digit_table_offset(size_t n) { return radix_temp_offset(n) + 2 * radix_temp_stride(n); }
inline size_t digit_table_bytes(size_t n) { return align_up(4 * 256 * ceil_div(n, kDigitTile), 256); }

struct LaunchOpts {
    uint64_t timeout_ns = 1000000000ull;  // a look-back wait gives up after this long
    bool skip_first_tile = false;        // test hook: no CTA ever takes tile 0
    // Status words of a persistent kernel, starting at word status_region of
    // the status area.  By default the kernel clears them itself behind its
    // start barrier; reset_status = false says they are clear already.  A
    // caller that runs many passes in a row (the radix split) has each pass
    // clear clear_words words from clear_region on for the next one, which
    // then needs neither a clear nor a barrier.
    bool reset_status = true;
    uint32_t status_region = 0, clear_region = 0, clear_words = 0;
};

// Clears the tile counter and `tiles` status words; then the kernel of the
// call can run.  With skip_first_tile the counter starts at 1 instead.
cudaError_t reset_tiles(uint8_t *ws, size_t tiles, cudaStream_t s, bool skip_first_tile);

// Clears the header words of the count pre-pass and the radix histogram
// (the header but its error word, start-barrier words and tile counter)
// before those kernels.
cudaError_t clear_accumulators(uint8_t *ws, cudaStream_t s);

// Launchers.  All arguments were validated by api.cu; n >= 1.
// carry (device, nullable): one element of dt added to every output and to
// the total.
cudaError_t launch_scan(const void *in, void *out, void *total, uint32_t n, gc_dtype dt,
                        uint8_t *ws, cudaStream_t s, const LaunchOpts &o, bool inclusive = false,
                        const void *carry = nullptr);

// A parameterised predicate as the kernels take it (see gcd::PredCmp): keep
// keys in [lo, lo + span] (xor invert), or (x & mask) == value (xor invert).
struct CmpSpec {
    uint32_t lo, span, invert, is_mask, mask, value;
};
cudaError_t launch_select_cmp(const void *in, void *out, uint32_t *count, uint32_t n, gc_dtype dt,
                              const CmpSpec &c, uint8_t *ws, cudaStream_t s, const LaunchOpts &o);
cudaError_t launch_partition_cmp(const void *in, void *out, uint32_t *count_true, uint32_t n,
                                 gc_dtype dt, const CmpSpec &c, uint8_t *ws, cudaStream_t s,
                                 const LaunchOpts &o);
// obase (device, nullable): survivors go to out[*obase + rank]; a run that
// would end past cap (elements of out) is refused on the device
// (GC_ERR_DEVICE_CHECK).  Without obase, cap is n.
cudaError_t launch_select(const void *in, void *out, uint32_t *count, uint32_t n, gc_dtype dt,
                          gc_pred p, uint8_t *ws, cudaStream_t s, const LaunchOpts &o,
                          const uint64_t *obase = nullptr, uint64_t cap = 0);
// per_tile: one atomic per tile (gc_select_if_atomic_tile); otherwise one
// per survivor (gc_select_if_atomic).
cudaError_t launch_select_atomic(const void *in, void *out, uint32_t *count, uint32_t n,
                                 gc_dtype dt, gc_pred p, cudaStream_t s, bool per_tile);
cudaError_t launch_partition(const void *in, void *out, uint32_t *count_true, uint32_t n,
                             gc_dtype dt, gc_pred p, uint8_t *ws, cudaStream_t s,
                             const LaunchOpts &o);
cudaError_t launch_split_radix(const uint32_t *keys_in, const uint32_t *vals_in,
                               uint32_t *keys_out, uint32_t *vals_out, uint32_t n, int begin_bit,
                               int end_bit, uint8_t *ws, cudaStream_t s, const LaunchOpts &o,
                               uint32_t key_neg = 0u, uint32_t key_flip = 0u);

// The pre-passes of a scan, select-if or partition split over shards, and
// the placed partition.  See gc_reduce, gc_count_if, gc_partition_at.
cudaError_t launch_reduce(const void *in, void *total, uint32_t n, gc_dtype dt, uint8_t *ws,
                          cudaStream_t s);
cudaError_t launch_count_if(const void *in, uint32_t *count, uint32_t n, gc_dtype dt, gc_pred p,
                            uint8_t *ws, cudaStream_t s);
cudaError_t launch_partition_at(const void *in, void *out, uint64_t capacity,
                                const uint64_t *offsets, uint32_t *count_true, uint32_t n,
                                gc_dtype dt, gc_pred p, uint8_t *ws, cudaStream_t s,
                                const LaunchOpts &o);
// One thread: the offsets of shard `rank` from the totals of all `parts`
// shards (gc_shard_offsets).
cudaError_t launch_shard_offsets(gc_op op, gc_dtype dt, const uint32_t *totals, uint32_t parts,
                                 uint32_t rank, uint64_t sizes_before, void *offsets,
                                 cudaStream_t s);

cudaError_t launch_radix_sort_digits(const uint32_t *keys_in, const uint32_t *vals_in,
                                     uint32_t *keys_out, uint32_t *vals_out, uint32_t n,
                                     uint32_t key_neg, uint32_t key_flip, uint8_t *ws,
                                     cudaStream_t s, const LaunchOpts &o);

uint32_t scan_tile_elems();
uint32_t select_tile_elems();
uint32_t partition_tile_elems();
uint32_t split_tile_elems();
uint32_t atomic_tile_elems();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count();  // multiprocessors of the current device (cached per device)

// Test hook (gc_testing_force_fallback): when set, every scan, select-if
// and partition runs the one-tile-per-CTA kernels, which otherwise run only
// when the device refuses a cooperative grid.
bool force_fallback();

// Grid of a persistent kernel: as many CTAs as fit on the device at once
// (never more than there are tiles).  Raises the kernel's dynamic shared
// memory limit to `smem` first.  Returns <= 0 on failure.
int persistent_grid(const void *kernel, int threads, size_t smem, uint32_t tiles);

}  // namespace gch
