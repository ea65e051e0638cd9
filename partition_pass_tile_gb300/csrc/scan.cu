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
#include <algorithm>

#include "gc_device.cuh"
#include "gc_internal.h"
#include "gc_launch.cuh"

namespace {

using namespace gcd;

template <int THREADS, int ROWS, bool VEC, bool LB, bool INCL>
__global__ void __launch_bounds__(THREADS)
scan_u32_kernel(const uint32_t *in, uint32_t *out, uint32_t *total, uint32_t n,
                uint32_t num_tiles, uint8_t *ws, uint64_t timeout_ns, const uint32_t *carry)
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
    if (carry != nullptr) prefix += *carry;  // the look-back itself stays carry-free
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
                uint32_t num_tiles, uint8_t *ws, double *prefix64, uint64_t timeout_ns,
                const uint32_t *carry)
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
    if (carry != nullptr) excl += double(__uint_as_float(*carry));
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

// Sum of the n elements, the aggregate half of the scan alone: the pre-pass
// of a scan split over shards, whose offsets need every shard's total before
// any shard is scanned.  Grid-stride 128-bit loads; int32 / uint32 add modulo
// 2^32, float32 sums each 4-vector in float and accumulates the vector sums
// per thread as a float pair (TwoSum), so the thread's error stays near one
// rounding of its total.  Each CTA stores its partial in the workspace's
// status area; the CTA that finishes last (ticket counter) adds the partials
// in CTA order (float32 in double) and writes the total, so the result does
// not depend on the order in which CTAs finish.
template <bool F32, bool VEC>
__global__ void __launch_bounds__(256)
reduce_kernel(const uint32_t *__restrict__ in, uint32_t n, uint8_t *ws, uint32_t *total)
{
    constexpr int W = 256 / 32;
    __shared__ float s_h[W], s_l[W];
    __shared__ uint32_t s_u[W];
    __shared__ uint32_t s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t nvec = (n + 3u) / 4u;
    const uint32_t stride = gridDim.x * 256u;
    uint32_t su = 0u;
    float h = 0.0f, l = 0.0f;
    constexpr uint32_t kUnroll = 4;  // loads in flight per thread
    for (uint32_t v0 = blockIdx.x * 256u + tid; v0 < nvec; v0 += kUnroll * stride) {
        uint32_t x[kUnroll][4];
#pragma unroll
        for (uint32_t u = 0; u < kUnroll; ++u) {
            const uint32_t v = v0 + u * stride;
            if (v < nvec) load4<VEC>(in, 4u * v, n, 0u, x[u]);
            else x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0u;
        }
#pragma unroll
        for (uint32_t u = 0; u < kUnroll; ++u) {
            if (F32) {
                const float a = (__uint_as_float(x[u][0]) + __uint_as_float(x[u][1])) +
                                (__uint_as_float(x[u][2]) + __uint_as_float(x[u][3]));
                ff_add(h, l, a, 0.0f, h, l);
            } else {
                su += x[u][0] + x[u][1] + x[u][2] + x[u][3];
            }
        }
    }
    uint64_t *partial = reinterpret_cast<uint64_t *>(ws + kStatusOff);
    if (F32) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(kFullMask, h, o), ol = __shfl_xor_sync(kFullMask, l, o);
            ff_add(h, l, oh, ol, h, l);
        }
        if (lane == 0) {
            s_h[warp] = h;
            s_l[warp] = l;
        }
    } else {
        su = warp_sum(su);
        if (lane == 0) s_u[warp] = su;
    }
    __syncthreads();
    if (tid == 0) {
        uint64_t word;
        if (F32) {
            float th = 0.0f, tl = 0.0f;
            for (int w = 0; w < W; ++w) ff_add(th, tl, s_h[w], s_l[w], th, tl);
            word = (uint64_t(__float_as_uint(tl)) << 32) | __float_as_uint(th);
        } else {
            uint32_t t = 0u;
            for (int w = 0; w < W; ++w) t += s_u[w];
            word = t;
        }
        st_relaxed_gpu(partial + blockIdx.x, word);
        __threadfence();
        s_last = atomicAdd(hdr_u32(ws, kHdrReduceCtr), 1u) == gridDim.x - 1u ? 1u : 0u;
    }
    __syncthreads();
    if (s_last == 0u) return;
    // The last CTA adds the partials, every thread a strided share, then the
    // CTA in warp order: a fixed order, so the total is the same every call.
    __threadfence();
    __shared__ double s_d[W];
    if (F32) {
        double acc = 0.0;
        for (uint32_t b = tid; b < gridDim.x; b += 256u) {
            const uint64_t w = ld_relaxed_gpu(partial + b);
            acc += double(__uint_as_float(uint32_t(w))) + double(__uint_as_float(uint32_t(w >> 32)));
        }
        acc = warp_sum(acc);
        if (lane == 0) s_d[warp] = acc;
    } else {
        uint32_t acc = 0u;
        for (uint32_t b = tid; b < gridDim.x; b += 256u) acc += uint32_t(ld_relaxed_gpu(partial + b));
        acc = warp_sum(acc);
        if (lane == 0) s_u[warp] = acc;
    }
    __syncthreads();
    if (tid == 0) {
        if (F32) {
            double t = 0.0;
            for (int w = 0; w < W; ++w) t += s_d[w];
            *total = __float_as_uint(float(t));
        } else {
            uint32_t t = 0u;
            for (int w = 0; w < W; ++w) t += s_u[w];
            *total = t;
        }
        atomicExch(hdr_u32(ws, kHdrReduceCtr), 0u);
    }
}

}  // namespace

namespace gch {

cudaError_t launch_reduce(const void *in, void *total, uint32_t n, gc_dtype dt, uint8_t *ws,
                          cudaStream_t s)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *t = static_cast<uint32_t *>(total);
    // Partials take one status word per CTA: never more CTAs than the
    // workspace has words for.
    const size_t want = ceil_div(ceil_div(n, 4), 256);
    size_t grid = std::min<size_t>(want, size_t(sm_count()) * 8);
    grid = std::max<size_t>(1, std::min(grid, max_tiles(n)));
    cudaError_t e = clear_accumulators(ws, s);
    if (e != cudaSuccess) return e;
    const bool vec = aligned16(in);
    if (dt == GC_F32) {
        if (vec) reduce_kernel<true, true><<<unsigned(grid), 256, 0, s>>>(i, n, ws, t);
        else reduce_kernel<true, false><<<unsigned(grid), 256, 0, s>>>(i, n, ws, t);
    } else {
        if (vec) reduce_kernel<false, true><<<unsigned(grid), 256, 0, s>>>(i, n, ws, t);
        else reduce_kernel<false, false><<<unsigned(grid), 256, 0, s>>>(i, n, ws, t);
    }
    return cudaGetLastError();
}

uint32_t scan_tile_elems() { return tile_elems(kScanPipeThreads, kScanPipeRows); }

namespace {

template <bool F32, bool OUT_VEC, bool INCL, bool SH = false>
cudaError_t launch_scan_pipe(const uint32_t *in, uint32_t *out, uint32_t *total, uint32_t n,
                             uint8_t *ws, cudaStream_t s, const LaunchOpts &o,
                             const uint32_t *carry)
{
    using Op = gcd::ScanOp<kScanPipeThreads, kScanPipeRows, F32, OUT_VEC, INCL, SH>;
    Op op{{in}, out, total, carry};
    return gcd::launch_pipeline<kScanPipeThreads, kScanPipeStages>(op, n, ws, s, o);
}

template <bool INCL>
cudaError_t launch_scan_impl(const void *in, void *out, void *total, uint32_t n, gc_dtype dt,
                             uint8_t *ws, cudaStream_t s, const LaunchOpts &o, const void *carry)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    auto *t = static_cast<uint32_t *>(total);
    auto *c = static_cast<const uint32_t *>(carry);
    cudaError_t e;
    if (!o.skip_first_tile && !force_fallback()) {
        const bool ov = aligned16(out);
        // An input that is not 16-byte aligned is staged shifted (and its
        // outputs stored element by element).
        if (!aligned16(in))
            e = dt == GC_F32 ? launch_scan_pipe<true, false, INCL, true>(i, u, t, n, ws, s, o, c)
                             : launch_scan_pipe<false, false, INCL, true>(i, u, t, n, ws, s, o, c);
        else if (dt == GC_F32)
            e = ov ? launch_scan_pipe<true, true, INCL>(i, u, t, n, ws, s, o, c)
                   : launch_scan_pipe<true, false, INCL>(i, u, t, n, ws, s, o, c);
        else
            e = ov ? launch_scan_pipe<false, true, INCL>(i, u, t, n, ws, s, o, c)
                   : launch_scan_pipe<false, false, INCL>(i, u, t, n, ws, s, o, c);
        if (e == cudaSuccess) return e;
        // The device cannot hold the whole cooperative grid right now (another
        // context holds SMs): fall through to the kernel that needs no
        // co-residency.  Clear the launch error first.
        (void)cudaGetLastError();
    }
    // A refused cooperative launch (or a test hook): one tile per CTA, loads
    // straight into registers.
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
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, prefix64, o.timeout_ns, c);
        else
            scan_f32_kernel<kScanThreads, kScanRows, false, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, prefix64, o.timeout_ns, c);
    } else {
        if (vec)
            scan_u32_kernel<kScanThreads, kScanRows, true, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, o.timeout_ns, c);
        else
            scan_u32_kernel<kScanThreads, kScanRows, false, kCtaLookback, INCL>
                <<<grid, kScanThreads, 0, s>>>(i, u, t, n, tiles, ws, o.timeout_ns, c);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const void *in, void *out, void *total, uint32_t n, gc_dtype dt,
                        uint8_t *ws, cudaStream_t s, const LaunchOpts &o, bool inclusive,
                        const void *carry)
{
    return inclusive ? launch_scan_impl<true>(in, out, total, n, dt, ws, s, o, carry)
                     : launch_scan_impl<false>(in, out, total, n, dt, ws, s, o, carry);
}

}  // namespace gch
