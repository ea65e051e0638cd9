// select.cu -- fused single-pass stable select-if, and the atomic-counter
// comparison path.
//
// Stable select-if is the three steps of "compaction.cu -- Day 33" (file
// header): predicate, exclusive scan of the 0/1 flags, scatter of survivors
// to out[rank].  "The CUDA Handbook, ch. 13: Stream compaction" (Listing
// 13-17) fuses them into one pass over tiles with a look-back on the tile
// keep counts and has the highest-numbered tile write the grand total.  This
// kernel does the same with GB300-shaped tiles:
//   1. 128-bit loads; the predicate of each thread's 4 elements per row
//      becomes a 4-bit mask and its popcount;
//   2. the per-row counts (at most 128 per warp and row, so 8 bits each) are
//      packed four to a word and scanned across the warp with shuffles: one
//      scan yields every lane's offset in four chunks at once;
//   3. warp 0 scans the chunk totals, publishes the tile's keep count, looks
//      back for the number kept by all earlier tiles, publishes its own
//      inclusive count; the last tile writes the grand total;
//   4. survivors are placed in shared memory at their rank within the tile,
//      shifted so that the shared and global addresses agree modulo 16 bytes,
//      and the CTA writes its survivors as one contiguous run with 128-bit
//      stores (scalar stores only for the partial vectors at the two ends).
// The input is read once; only survivors and the count are written.
#include <algorithm>

#include "gc_device.cuh"
#include "gc_internal.h"
#include "gc_launch.cuh"


namespace {

using namespace gcd;

template <class Pred, int THREADS, int ROWS, bool VEC, bool LB>
__global__ void __launch_bounds__(THREADS)
select_kernel(const uint32_t *__restrict__ in, uint32_t *__restrict__ out, uint32_t *count,
              uint32_t n, uint32_t num_tiles, Pred pred, uint8_t *ws, uint64_t timeout_ns,
              SelectPlacement place)
{
    using TT = Tile<THREADS, ROWS>;
    __shared__ uint32_t s_tile;
    __shared__ uint32_t s_chunk[TT::kChunks];
    __shared__ PrefixSmem s_ps;
    __shared__ __align__(16) uint32_t s_buf[TT::kElems + 4];

    const uint32_t tile = claim_tile(ws, &s_tile);
    if (tile >= num_tiles) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t base = tile * uint32_t(TT::kElems);

    uint32_t x[ROWS][4];
    uint32_t mask[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const uint32_t idx = base + r * TT::kRowElems + 4 * tid;
        load4<VEC>(in, idx, n, 0u, x[r]);
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) m |= uint32_t(idx + k < n && pred(x[r][k])) << k;
        mask[r] = m;
    }

    uint32_t lane_excl[ROWS];
    rank_masks<TT>(mask, lane_excl, s_chunk);
    __syncthreads();

    uint32_t prefix, kept;
    resolve_prefix_u32<TT, LB>(s_chunk, tile, ws, timeout_ns, s_ps, prefix, kept);
    if (tid == 0 && tile == num_tiles - 1) *count = prefix + kept;
    // survivors go to out[obase + prefix + rank] (obase = 0 unless placed)
    const uint64_t ob = place.obase != nullptr ? *place.obase : 0ull;
    if (ob + uint64_t(prefix) + kept > place.cap) {
        if (tid == 0) record_error(ws, kDeviceCheckCode, tile);
        return;
    }
    out += ob & ~3ull;
    const uint32_t out_base = uint32_t(ob & 3ull) + prefix;
    const uint32_t shift = VEC ? (out_base & 3u) : 0u;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        uint32_t pos = shift + s_chunk[r * TT::kWarps + warp] + lane_excl[r];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if ((mask[r] >> k) & 1u) s_buf[pos++] = x[r][k];
        }
    }
    __syncthreads();
    store_run<THREADS, VEC>(out, out_base, s_buf, shift, kept);
}

// The comparison path as "compaction.cu -- Day 33" writes it (compactAtomic):
// one pass over the input, and every survivor takes its output slot with one
// atomicAdd on the single counter the whole grid shares, then writes itself
// there.  No scan and no order: where a survivor lands depends on the order
// in which the atomics resolve.  The counter is cleared on the stream before
// the launch (the page's zeroCount).  The grid is a fixed number of CTAs per
// SM that stride over the input, 16 bytes per thread per step, so the loads
// stay coalesced; the stores are single elements at whatever slots the
// atomics return.
template <class Pred, bool VEC>
__global__ void __launch_bounds__(256)
select_atomic_elem_kernel(const uint32_t *__restrict__ in, uint32_t *__restrict__ out,
                          uint32_t *count, uint32_t n, Pred pred)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t tail = 0u;  // elements before this index went through the vector loop
    if (VEC) {
        const uint32_t nvec = n >> 2;
        for (uint32_t v = first; v < nvec; v += stride) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(in) + v);
            const uint32_t x[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (pred(x[k])) out[atomicAdd(count, 1u)] = x[k];
        }
        tail = nvec << 2;
    }
    for (uint32_t i = tail + first; i < n; i += stride) {
        const uint32_t x = __ldcs(in + i);
        if (pred(x)) out[atomicAdd(count, 1u)] = x;
    }
}

// The same comparison with one atomic per tile instead of one per survivor:
// each CTA ranks its tile's survivors (as select_kernel does), claims a run
// of that many output slots with one atomicAdd on the shared counter, and
// writes its survivors there as one contiguous run; which CTA reaches the
// counter first decides where its run lands.
template <class Pred, int THREADS, int ROWS, bool VEC>
__global__ void __launch_bounds__(THREADS)
select_atomic_kernel(const uint32_t *__restrict__ in, uint32_t *__restrict__ out,
                     uint32_t *count, uint32_t n, Pred pred)
{
    using TT = Tile<THREADS, ROWS>;
    __shared__ uint32_t s_chunk[TT::kChunks];
    __shared__ uint32_t s_base, s_kept;
    __shared__ __align__(16) uint32_t s_buf[TT::kElems + 4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = blockIdx.x * uint32_t(TT::kElems);

    uint32_t x[ROWS][4], mask[ROWS], lane_excl[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const uint32_t idx = base + r * TT::kRowElems + 4 * tid;
        load4<VEC>(in, idx, n, 0u, x[r]);
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) m |= uint32_t(idx + k < n && pred(x[r][k])) << k;
        mask[r] = m;
    }
    rank_masks<TT>(mask, lane_excl, s_chunk);
    __syncthreads();
    if (warp == 0) {
        const uint32_t kept = scan_chunks_warp0<TT>(s_chunk);
        if (lane == 0) {
            s_kept = kept;
            s_base = kept != 0u ? atomicAdd(count, kept) : 0u;
        }
    }
    __syncthreads();
    const uint32_t kept = s_kept, out_base = s_base;
    if (kept == 0u) return;
    const uint32_t shift = VEC ? (out_base & 3u) : 0u;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        uint32_t pos = shift + s_chunk[r * TT::kWarps + warp] + lane_excl[r];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if ((mask[r] >> k) & 1u) s_buf[pos++] = x[r][k];
    }
    __syncthreads();
    store_run<THREADS, VEC>(out, out_base, s_buf, shift, kept);
}

template <class Pred>
cudaError_t dispatch_select(const uint32_t *in, uint32_t *out, uint32_t *count, uint32_t n,
                            Pred pred, uint8_t *ws, cudaStream_t s, const gch::LaunchOpts &o,
                            SelectPlacement place)
{
    if (!o.skip_first_tile && !gch::force_fallback()) {
        constexpr int PT = gch::kSelectPipeThreads, PR = gch::kSelectPipeRows;
        constexpr int PS = gch::kSelectPipeStages;
        // The placed form (a shard of a larger select-if) is its own
        // instantiation, so the plain select keeps its 32-bit addressing.
        auto go = [&](auto op) {
            op.srcs[0] = in;
            op.out = out;
            op.count = count;
            op.pred = pred;
            op.place = place;
            op.ws = ws;
            return gcd::launch_pipeline<PT, PS>(op, n, ws, s, o);
        };
        const bool vec = gch::aligned16(out), placed = place.obase != nullptr;
        cudaError_t e;
        if (!gch::aligned16(in))  // staged shifted, survivors stored element by element
            e = placed ? go(gcd::SelectOp<PT, PR, Pred, false, true, true>{})
                       : go(gcd::SelectOp<PT, PR, Pred, false, false, true>{});
        else if (placed)
            e = vec ? go(gcd::SelectOp<PT, PR, Pred, true, true>{}) : go(gcd::SelectOp<PT, PR, Pred, false, true>{});
        else
            e = vec ? go(gcd::SelectOp<PT, PR, Pred, true, false>{}) : go(gcd::SelectOp<PT, PR, Pred, false, false>{});
        if (e == cudaSuccess) return e;
        (void)cudaGetLastError();  // cooperative grid refused: one tile per CTA instead
    }
    constexpr int T = gch::kSelectThreads, R = gch::kSelectRows;
    const uint32_t tiles = uint32_t(gch::ceil_div(n, gch::tile_elems(T, R)));
    cudaError_t e = gch::reset_tiles(ws, tiles, s, o.skip_first_tile);
    if (e != cudaSuccess) return e;
    const uint32_t grid = o.skip_first_tile ? tiles - 1 : tiles;
    if (grid == 0) return cudaSuccess;
    if (gch::aligned16(in) && gch::aligned16(out))
        select_kernel<Pred, T, R, true, gch::kCtaLookback><<<grid, T, 0, s>>>(in, out, count, n, tiles, pred, ws, o.timeout_ns, place);
    else
        select_kernel<Pred, T, R, false, gch::kCtaLookback><<<grid, T, 0, s>>>(in, out, count, n, tiles, pred, ws, o.timeout_ns, place);
    return cudaGetLastError();
}

template <class Pred>
cudaError_t dispatch_atomic_tile(const uint32_t *in, uint32_t *out, uint32_t *count, uint32_t n,
                                 Pred pred, cudaStream_t s)
{
    constexpr int T = gch::kAtomicThreads, R = gch::kAtomicRows;
    const uint32_t tiles = uint32_t(gch::ceil_div(n, gch::tile_elems(T, R)));
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    if (gch::aligned16(in) && gch::aligned16(out))
        select_atomic_kernel<Pred, T, R, true><<<tiles, T, 0, s>>>(in, out, count, n, pred);
    else
        select_atomic_kernel<Pred, T, R, false><<<tiles, T, 0, s>>>(in, out, count, n, pred);
    return cudaGetLastError();
}

template <class Pred>
cudaError_t dispatch_atomic_elem(const uint32_t *in, uint32_t *out, uint32_t *count, uint32_t n,
                                 Pred pred, cudaStream_t s)
{
    constexpr int T = 256;
    // Enough CTAs to keep every SM's loads in flight; each thread then
    // strides over the input.
    const uint32_t want = uint32_t(gch::sm_count()) * 8u;
    const uint32_t grid = uint32_t(std::max<size_t>(1, std::min<size_t>(want, gch::ceil_div(n, 4 * T))));
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    if (gch::aligned16(in))
        select_atomic_elem_kernel<Pred, true><<<grid, T, 0, s>>>(in, out, count, n, pred);
    else
        select_atomic_elem_kernel<Pred, false><<<grid, T, 0, s>>>(in, out, count, n, pred);
    return cudaGetLastError();
}

template <class Pred>
cudaError_t dispatch_atomic(const uint32_t *in, uint32_t *out, uint32_t *count, uint32_t n,
                            Pred pred, cudaStream_t s, bool per_tile)
{
    return per_tile ? dispatch_atomic_tile(in, out, count, n, pred, s)
                    : dispatch_atomic_elem(in, out, count, n, pred, s);
}

}  // namespace

namespace gch {

uint32_t select_tile_elems() { return tile_elems(kSelectPipeThreads, kSelectPipeRows); }
uint32_t atomic_tile_elems() { return tile_elems(kAtomicThreads, kAtomicRows); }

cudaError_t launch_select(const void *in, void *out, uint32_t *count, uint32_t n, gc_dtype dt,
                          gc_pred p, uint8_t *ws, cudaStream_t s, const LaunchOpts &o,
                          const uint64_t *obase, uint64_t cap)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    const gcd::SelectPlacement place{obase, obase != nullptr ? cap : uint64_t(n)};
    switch (p) {
    case GC_PRED_NONZERO:
        if (dt == GC_F32) return dispatch_select(i, u, count, n, gcd::PredNonzeroF32{}, ws, s, o, place);
        return dispatch_select(i, u, count, n, gcd::PredNonzeroInt{}, ws, s, o, place);
    case GC_PRED_ODD: return dispatch_select(i, u, count, n, gcd::PredOdd{}, ws, s, o, place);
    default: return dispatch_select(i, u, count, n, gcd::PredEven{}, ws, s, o, place);
    }
}

cudaError_t launch_select_cmp(const void *in, void *out, uint32_t *count, uint32_t n, gc_dtype dt,
                              const CmpSpec &c, uint8_t *ws, cudaStream_t s, const LaunchOpts &o)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    const gcd::SelectPlacement place{nullptr, uint64_t(n)};
    if (dt == GC_I32)
        return dispatch_select(i, u, count, n, gcd::PredCmp<0>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o, place);
    if (dt == GC_U32)
        return dispatch_select(i, u, count, n, gcd::PredCmp<1>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o, place);
    return dispatch_select(i, u, count, n, gcd::PredCmp<2>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o, place);
}

cudaError_t launch_select_atomic(const void *in, void *out, uint32_t *count, uint32_t n,
                                 gc_dtype dt, gc_pred p, cudaStream_t s, bool per_tile)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    switch (p) {
    case GC_PRED_NONZERO:
        if (dt == GC_F32) return dispatch_atomic(i, u, count, n, gcd::PredNonzeroF32{}, s, per_tile);
        return dispatch_atomic(i, u, count, n, gcd::PredNonzeroInt{}, s, per_tile);
    case GC_PRED_ODD: return dispatch_atomic(i, u, count, n, gcd::PredOdd{}, s, per_tile);
    default: return dispatch_atomic(i, u, count, n, gcd::PredEven{}, s, per_tile);
    }
}

}  // namespace gch
