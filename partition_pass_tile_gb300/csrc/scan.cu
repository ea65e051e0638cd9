// scan.cu -- single-pass exclusive scan (int32 / uint32 / float32).
//
// out[i] = in[0] + ... + in[i-1], out[0] = 0: the exclusive scan of
// "scan_2.cu -- Day 32: the work-efficient scan" (scanExclusiveCpu) and the
// "rank[i] becomes the number of survivors before i" step of
// "compaction.cu -- Day 33".  Those pages reach it with three or five
// launches (tile scan, scan of tile sums, add-back); here one launch reads
// every element once and writes it once, and tiles exchange only their
// totals through the decoupled look-back of gc_device.cuh.
//
// Per tile (THREADS x ROWS vectors of 4):
//   1. 128-bit loads, each thread sums its 4 elements of each row;
//   2. a shuffle scan across the warp gives each lane's offset within its
//      chunk (a warp's 128 elements of one row); lane 31 leaves the chunk
//      total in shared memory;
//   3. warp 0 scans the chunk totals, publishes the tile total, looks back
//      for the tile's exclusive prefix and publishes the inclusive one;
//   4. every thread adds prefix + chunk offset + lane offset + running
//      in-thread sum and writes 128-bit vectors at the same positions.
// In place (in == out) is safe: each element is read before the barriers
// and written after them by the same thread, and no thread touches another
// thread's elements.
#include "gc_device.cuh"
#include "gc_internal.h"
#include "gc_launch.cuh"

namespace {

using namespace gcd;

template <int THREADS, int ROWS, bool VEC, bool LB, bool INCL>
__global__ void __launch_bounds__(THREADS)
scan_u32_kernel(const uint32_t *in, uint32_t *out, uint32_t *total, uint32_t n,
                uint32_t num_tiles, uint8_t *ws, uint64_t timeout_ns)
{
    using TT = Tile<THREADS, ROWS>;
    __shared__ uint32_t s_tile;
    __shared__ uint32_t s_chunk[TT::kChunks];
    __shared__ PrefixSmem s_ps;

    const uint32_t tile = claim_tile(ws, &s_tile);
    if (tile >= num_tiles) return;  // only with the skip-first-tile test hook
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = tile * uint32_t(TT::kElems);

    uint32_t x[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        load4<VEC>(in, base + r * TT::kRowElems + 4 * tid, n, 0u, x[r]);

    uint32_t lane_excl[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const uint32_t s = x[r][0] + x[r][1] + x[r][2] + x[r][3];
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
        }
        lane_excl[r] = incl - s;
        if (lane == 31) s_chunk[r * TT::kWarps + warp] = incl;
    }
    __syncthreads();

    uint32_t prefix, agg;
    resolve_prefix_u32<TT, LB>(s_chunk, tile, ws, timeout_ns, s_ps, prefix, agg);
    if (tid == 0 && total != nullptr && tile == num_tiles - 1) *total = prefix + agg;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        uint32_t v = prefix + s_chunk[r * TT::kWarps + warp] + lane_excl[r];
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (INCL) v += x[r][k];
            o[k] = v;
            if (!INCL) v += x[r][k];
        }
        store4<VEC>(out, base + r * TT::kRowElems + 4 * tid, n, o);
    }
}

// float32: the same structure.  Inside the tile the sums are float32; the
// tile's exclusive prefix arrives as a double and is split into a float pair
// hi + lo (hi = the double rounded to float, lo = the remainder rounded to
// float), and each output is hi + (lo + local).  The carry between tiles
// therefore never rounds to float32 before the last add of each element.
template <int THREADS, int ROWS, bool VEC, bool LB, bool INCL>
__global__ void __launch_bounds__(THREADS)
scan_f32_kernel(const uint32_t *in_bits, uint32_t *out_bits, uint32_t *total_bits, uint32_t n,
                uint32_t num_tiles, uint8_t *ws, double *prefix64, uint64_t timeout_ns)
{
    using TT = Tile<THREADS, ROWS>;
    __shared__ uint32_t s_tile;
    __shared__ float s_chunk[TT::kChunks];
    __shared__ PrefixSmem s_ps;

    const uint32_t tile = claim_tile(ws, &s_tile);
    if (tile >= num_tiles) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = tile * uint32_t(TT::kElems);

    uint32_t raw[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        load4<VEC>(in_bits, base + r * TT::kRowElems + 4 * tid, n, 0u, raw[r]);

    float lane_excl[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const float s = (__uint_as_float(raw[r][0]) + __uint_as_float(raw[r][1])) +
                        (__uint_as_float(raw[r][2]) + __uint_as_float(raw[r][3]));
        float incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
        }
        float ex = __shfl_up_sync(kFullMask, incl, 1);
        lane_excl[r] = (lane == 0) ? 0.0f : ex;
        if (lane == 31) s_chunk[r * TT::kWarps + warp] = incl;
    }
    __syncthreads();

    double excl;
    float agg;
    resolve_prefix_f32<TT, LB>(s_chunk, tile, ws, prefix64, timeout_ns, s_ps, excl, agg);
    if (tid == 0 && total_bits != nullptr && tile == num_tiles - 1)
        *total_bits = __float_as_uint(float(excl + double(agg)));
    const float hi = float(excl);
    const float lo = float(excl - double(hi));
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        float local = s_chunk[r * TT::kWarps + warp] + lane_excl[r];
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (INCL) local += __uint_as_float(raw[r][k]);
            o[k] = __float_as_uint(hi + (lo + local));
            if (!INCL) local += __uint_as_float(raw[r][k]);
        }
        store4<VEC>(out_bits, base + r * TT::kRowElems + 4 * tid, n, o);
    }
}

}  // namespace

namespace gch {

uint32_t scan_tile_elems() { return tile_elems(kScanPipeThreads, kScanPipeRows); }

namespace {

template <bool F32, bool OUT_VEC, bool INCL>
cudaError_t launch_scan_pipe(const uint32_t *in, uint32_t *out, uint32_t *total, uint32_t n,
                             uint8_t *ws, cudaStream_t s, const LaunchOpts &o)
{
    using Op = gcd::ScanOp<kScanPipeThreads, kScanPipeRows, F32, OUT_VEC, INCL>;
    Op op{{in}, out, total};
    return gcd::launch_pipeline<kScanPipeThreads, kScanPipeStages>(op, n, ws, s, o);
}

template <bool INCL>
cudaError_t launch_scan_impl(const void *in, void *out, void *total, uint32_t n, gc_dtype dt,
                             uint8_t *ws, cudaStream_t s, const LaunchOpts &o)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    auto *t = static_cast<uint32_t *>(total);
    cudaError_t e;
    if (aligned16(in) && !o.skip_first_tile) {
        const bool ov = aligned16(out);
        if (dt == GC_F32)
            e = ov ? launch_scan_pipe<true, true, INCL>(i, u, t, n, ws, s, o)
                   : launch_scan_pipe<true, false, INCL>(i, u, t, n, ws, s, o);
        else
            e = ov ? launch_scan_pipe<false, true, INCL>(i, u, t, n, ws, s, o)
                   : launch_scan_pipe<false, false, INCL>(i, u, t, n, ws, s, o);
        if (e == cudaSuccess) return e;
        // The device cannot hold the whole cooperative grid right now (another
        // context holds SMs): fall through to the kernel that needs no
        // co-residency.  Clear the launch error first.
        (void)cudaGetLastError();
    }
    // Unaligned input (or the test hook): one tile per CTA, loads straight
    // into registers.
    const uint32_t tile = tile_elems(kScanThreads, kScanRows);
    const uint32_t tiles = uint32_t(ceil_div(n, tile));
    e = reset_tiles(ws, tiles, s, o.skip_first_tile);
    if (e != cudaSuccess) return e;
    const bool vec = aligned16(in) && aligned16(out);
    const uint32_t grid = o.skip_first_tile ? tiles - 1 : tiles;
    if (grid == 0) return cudaSuccess;
    if (dt == GC_F32) {
        double *prefix64 = reinterpret_cast<double *>(ws + kHeaderBytes + status_bytes(tiles));
        if (vec)
            scan_f32_kernel<kScanThreads, kScanRows, true, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, prefix64, o.timeout_ns);
        else
            scan_f32_kernel<kScanThreads, kScanRows, false, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, prefix64, o.timeout_ns);
    } else {
        if (vec)
            scan_u32_kernel<kScanThreads, kScanRows, true, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, o.timeout_ns);
        else
            scan_u32_kernel<kScanThreads, kScanRows, false, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, o.timeout_ns);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const void *in, void *out, void *total, uint32_t n, gc_dtype dt,
                        uint8_t *ws, cudaStream_t s, const LaunchOpts &o, bool inclusive)
{
    return inclusive ? launch_scan_impl<true>(in, out, total, n, dt, ws, s, o)
                     : launch_scan_impl<false>(in, out, total, n, dt, ws, s, o);
}

}  // namespace gch
