// gc_tiles.cuh -- the persistent, pipelined single-pass tile driver shared by
// every 16-byte-aligned kernel of libgc, and the per-operation tile bodies
// (exclusive scan, select-if, partition / one-bit split).
//
// Every operation of the path has the same two halves ("compaction.cu --
// Day 33", file header: predicate, scan, scatter): a tile's aggregate (its
// sum, or how many elements its predicate keeps), and the tile's output once
// the aggregates of all earlier tiles are known (its exclusive prefix).  The
// driver runs them as a software pipeline over the tiles a CTA owns:
//
//   grid      cooperative (every CTA resident); CTA c of G owns tiles c,
//             c + G, c + 2G, ...
//   loads     TMA bulk copies into STAGES shared-memory stage buffers
//             (gc_pipe.cuh), issued as soon as a stage is free;
//   iteration k, t = the CTA's k-th tile, p = t - G its previous one:
//     1. issue the loads of p's window: the aggregates of tiles p - G + 1 ..
//        p - 1, which their CTAs published a whole iteration earlier;
//     2. reduce t in shared memory and publish its aggregate at once;
//     3. finish the window: prefix(p) = run + window, run = prefix(p) +
//        agg(p), where run is the inclusive prefix of the tile before p
//        (kept by the CTA, so the walk never goes past it);
//     4. op.finish: compute and write p's outputs, then re-arm p's stage.
//   No tile ever waits on another CTA for more than a reduction, and the
//   window loads are in flight during the reduction.
//
// This is the single-pass scan with decoupled look-back of "The CUDA
// Handbook, ch. 13: Stream compaction" (Listing 13-17 and the scan it builds
// on) with two changes for a GPU whose HBM wants megabytes in flight: tiles
// are owned round-robin and prefetched by TMA, and every look-back stops at
// the CTA's own previous tile, one iteration late, so it is one round of
// reads of already-published words.
#pragma once

#include <cstdint>
#include <type_traits>

#include "gc_device.cuh"
#include "gc_pipe.cuh"

namespace gcd {

// ---------------------------------------------------------------- float-float sums
// Error-free transformation of a + b (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Knuth's FastTwoSum, for |a| >= |b|: renormalises a float pair.
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e)
{
    s = a + b;
    e = b - (s - a);
}

// (ah + al) + (bh + bl) as a normalised float pair (double-float addition).
__device__ __forceinline__ void ff_add(float ah, float al, float bh, float bl, float &sh, float &sl)
{
    float s, e;
    two_sum(ah, bh, s, e);
    e += al + bl;
    fast_two_sum(s, e, sh, sl);
}

// Window of float32 aggregates summed in float32, per thread, across the
// warp (a butterfly) and across the CTA; every thread gets the sum.  At most
// two adds per thread, five in the warp and W - 1 across warps: the relative
// error of the window stays below about 14 float32 roundings (1e-6), and the
// window is added to a running prefix that is carried as a float pair, so
// the error does not grow with the number of tiles.
template <int THREADS>
__device__ __forceinline__ float window_finish_f32(const uint64_t *status, uint32_t lo, uint32_t hi,
                                                   WindowLoads &wl, uint8_t *ws, uint32_t tile,
                                                   uint64_t timeout_ns, float *s_win)
{
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < kWinPerThread; ++i) {
        const uint32_t j = lo + threadIdx.x + uint32_t(i) * THREADS;
        if (j < hi) {
            uint32_t v = uint32_t(wl.w[i]);
            if (uint32_t(wl.w[i] >> 32) == kFlagNone) v = await_aggregate(status, j, ws, tile, timeout_ns);
            sum += __uint_as_float(v);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
    if ((threadIdx.x & 31) == 0) s_win[threadIdx.x >> 5] = sum;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) t += s_win[w];
    return t;
}

// ---------------------------------------------------------------- the driver
//
// Per iteration (t = this CTA's k-th tile, p = its previous one):
//   window loads for p issued;
//   op.reduce(t): predicate / sums, in-tile ranks, one barrier, then every
//     warp derives the tile total and its own chunk offsets; the aggregate is
//     published and the per-thread offsets (and masks) are carried to t's
//     finish one iteration later;
//   op.load(p): p's elements into registers;
//   window finish (one barrier, which also orders every read of p's stage
//     before the writes op.finish may make into it);
//   op.finish(p): outputs from the carried offsets;
//   a barrier, then p's stage is re-armed.
// Where a persistent call's status words are (word offset from the status
// area), whether the kernel clears them itself first (behind the start
// barrier; otherwise they are clear already), and which words, unused by
// this call, it clears for the call after it.
struct StatusPlan {
    uint32_t region, self_clear, clear_region, clear_words;
};

template <int THREADS, int STAGES, class Op>
__device__ __forceinline__ void pipeline_run(const Op &op, uint8_t *smem, uint32_t n,
                                             uint32_t num_tiles, uint8_t *ws, uint64_t timeout_ns,
                                             const StatusPlan &plan)
{
    static_assert(STAGES >= 3, "the tile being reduced, the tile being finished, one in flight");
    static_assert(THREADS >= 32 * kBulkIssuers, "a warp per bulk-store issuer");
    using P = typename Op::template PipeT<STAGES>;
    constexpr uint32_t TE = Op::kTileElems;
    constexpr int W = THREADS / 32;
    __shared__ uint32_t s_win_u[W];
    __shared__ float s_win_hi[W];
    P pipe{smem};
#pragma unroll
    for (int a = 0; a < int(sizeof(op.srcs) / sizeof(op.srcs[0])); ++a)
        pipe.sh[a] = uint32_t(reinterpret_cast<uintptr_t>(op.srcs[a]) >> 2) & 3u;
    const int tid = threadIdx.x;
    uint64_t *status = reinterpret_cast<uint64_t *>(ws + kStatusOff) + plan.region;

    const bool self_clear = plan.self_clear != 0u;
    uint32_t epoch = 0u;  // thread 0: the start barrier's epoch, read before arriving
    if (tid == 0 && self_clear) epoch = bar_epoch(ws);
    if (tid == 0) pipe.init();
    __syncthreads();
    if (tid == 0) pipe.prime(op.srcs, TE, n, num_tiles);
    if (plan.clear_words != 0u) {
        // The next pass's words, which no tile of this pass reads or writes.
        uint64_t *next = reinterpret_cast<uint64_t *>(ws + kStatusOff) + plan.clear_region;
        for (uint32_t j = blockIdx.x * THREADS + tid; j < plan.clear_words; j += gridDim.x * THREADS)
            next[j] = 0ull;
    }
    bool bar_pending = false;  // thread 0: arrived, the barrier not yet seen complete
    if (self_clear) {
        // This call's own words, while the primed loads are in flight.
        for (uint32_t j = blockIdx.x * THREADS + tid; j < num_tiles; j += gridDim.x * THREADS)
            status[j] = 0ull;
        __syncthreads();
        if (tid == 0) bar_pending = !bar_arrive(ws, epoch);
    }

    uint32_t run_u = 0u;     // inclusive prefix of the tile before the previous one
    float run_h = 0.0f, run_l = 0.0f;  // the same for float32, as a float pair
    op.seed(run_u, run_h, run_l);      // a scan's carry-in, where it has one
    uint32_t prev_agg = 0u;  // aggregate bits of the previous tile
    typename Op::Carry cur{}, prv{};  // per-thread results of a reduction kept for its finish

    // Iteration 0, peeled: the CTA's first tile is reduced while the start
    // barrier completes, and its aggregate is published once it has.
    if (blockIdx.x >= num_tiles) {
        if (tid == 0 && bar_pending) bar_wait(ws, epoch, timeout_ns);
        return;
    }
    {
        const uint32_t tile = blockIdx.x;
        mbar_wait(pipe.bar(0), 0u, ws, timeout_ns);
        const uint32_t staged = staged_elems(tile, TE, n);
        uint32_t first_bits = 0u;
        auto publish = [&](uint32_t bits) {
            if (tid == 0) {
                if (self_clear)
                    first_bits = bits;
                else
                    publish_aggregate(status, tile, bits);
            }
        };
        if (staged == TE)
            prev_agg = op.template reduce<true>(pipe, 0, tile * TE, staged, n, cur, publish);
        else
            prev_agg = op.template reduce<false>(pipe, 0, tile * TE, staged, n, cur, publish);
        if (self_clear) {
            if (tid == 0) {
                if (bar_pending) bar_wait(ws, epoch, timeout_ns);
                publish_aggregate(status, tile, first_bits);
            }
            __syncthreads();  // every thread's first status read comes after the barrier
        }
        prv = cur;
    }
    for (uint32_t k = 1;; ++k) {
        const uint32_t tile = blockIdx.x + k * gridDim.x;
        const bool have = tile < num_tiles;
        const bool have_prev = true;
        const uint32_t prev = tile - gridDim.x;

        WindowLoads wl;
        if (have_prev) window_issue<THREADS>(status, window_lo(prev), prev, wl);

        uint32_t agg = 0u;
        if (have) {
            const int s = int(k % STAGES);
            mbar_wait(pipe.bar(s), (k / STAGES) & 1u, ws, timeout_ns);
            const uint32_t base = tile * TE;
            const uint32_t staged = staged_elems(tile, TE, n);
            // Publishes t's aggregate: every op calls it once, as soon as it is known.
            auto publish = [&](uint32_t bits) {
                if (tid == 0) publish_aggregate(status, tile, bits);
            };
            if (staged == TE)
                agg = op.template reduce<true>(pipe, s, base, staged, n, cur, publish);
            else
                agg = op.template reduce<false>(pipe, s, base, staged, n, cur, publish);
        }

        if (have_prev) {
            const int ps = int((k - 1) % STAGES);
            const uint32_t pbase = prev * TE;
            const uint32_t pstaged = staged_elems(prev, TE, n);
            const bool full = pstaged == TE;
            const bool last = prev == num_tiles - 1;
            typename Op::Loaded ld;
            if constexpr (Op::kPreload) {
                if (full)
                    op.template load<true>(pipe, ps, pbase, pstaged, n, prev_agg, ld);
                else
                    op.template load<false>(pipe, ps, pbase, pstaged, n, prev_agg, ld);
            }
            if constexpr (Op::kF32) {
                const float wsum = window_finish_f32<THREADS>(status, window_lo(prev), prev, wl, ws,
                                                              prev, timeout_ns, s_win_hi);
                float ph, pl;
                ff_add(run_h, run_l, wsum, 0.0f, ph, pl);  // prefix(p) = run + window
                ff_add(ph, pl, __uint_as_float(prev_agg), 0.0f, run_h, run_l);
                if (full)
                    op.template finish_f32<true>(pipe, ps, pbase, pstaged, n, ph, pl, last, run_h + run_l, prv, ld);
                else
                    op.template finish_f32<false>(pipe, ps, pbase, pstaged, n, ph, pl, last, run_h + run_l, prv, ld);
            } else {
                uint32_t wsum_u;
                double unused;
                window_finish<THREADS, false>(status, window_lo(prev), prev, wl, ws, prev, timeout_ns,
                                              s_win_u, nullptr, wsum_u, unused);
                const uint32_t prefix = run_u + wsum_u;
                run_u = prefix + prev_agg;
                if (full)
                    op.template finish<true>(pipe, ps, prev, pbase, pstaged, n, prefix, prev_agg, last, prv, ld);
                else
                    op.template finish<false>(pipe, ps, prev, pbase, pstaged, n, prefix, prev_agg, last, prv, ld);
            }
            bulk_issuers_wait_read();  // the stage's bulk stores have read it ...
            __syncthreads();           // ... and every thread is done with it
            if (tid == 0) pipe.refill(ps, op.srcs, prev, TE, n, num_tiles);
        }
        if (!have) break;
        prev_agg = agg;
        prv = cur;
    }
    bulk_issuers_wait_all();  // shared memory stays until the stores are done
}

// Grid limit of pipeline_run: the window of a tile must fit kWinPerThread
// loads per thread.
template <int THREADS>
constexpr int pipeline_max_grid() { return kWinPerThread * THREADS + 1; }

// ---------------------------------------------------------------- tile bodies

// The stage buffer as an op reads it: the shifted view when its input may
// not be 16-byte aligned (SH), the buffer itself otherwise.
template <bool SH, class P>
__device__ __forceinline__ uint32_t *stage_rd(const P &pipe, int s, int array = 0)
{
    if constexpr (SH) return pipe.rbuf(s, array);
    else return pipe.buf(s, array);
}

// The vectors of one staged tile.
template <class TT, bool FULL, bool SH = false>
__device__ __forceinline__ void tile_vectors(const uint32_t *sbuf, const uint32_t *gin,
                                             uint32_t base, uint32_t staged, uint32_t n,
                                             uint32_t (&x)[TT::kRows][4])
{
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r)
        stage_load4<FULL, SH>(sbuf, gin, base, r * TT::kRowElems + 4 * threadIdx.x, staged, n, 0u, x[r]);
}

// Exclusive scan, uint32 (int32 bits) or float32.
template <int THREADS, int ROWS, bool F32, bool OUT_VEC, bool INCL = false, bool SH = false>
struct ScanOp {
    using TT = Tile<THREADS, ROWS>;
    static constexpr uint32_t kTileElems = TT::kElems;
    static constexpr bool kF32 = F32;
    template <int STAGES>
    using PipeT = Pipe<kTileElems * 4u, STAGES, 1>;

    const uint32_t *srcs[1];
    uint32_t *out;
    uint32_t *total;
    const uint32_t *carry;  // device, nullable: a value of the dtype added to every output

    struct Carry {};
    static constexpr bool kPreload = false;
    struct Loaded {};

    // The running prefix before the first tile: the carry-in, or 0.
    __device__ __forceinline__ void seed(uint32_t &u, float &h, float &l) const
    {
        if (carry != nullptr) {
            const uint32_t c = *carry;
            u = c;
            h = __uint_as_float(c);
            l = 0.0f;
        }
    }

    template <bool FULL, class P>
    __device__ __forceinline__ void load(const P &, int, uint32_t, uint32_t, uint32_t, uint32_t,
                                         Loaded &) const {}

    // The aggregate only: a plain sum, so it is published as early as possible.
    template <bool FULL, class P, class Publish>
    __device__ __forceinline__ uint32_t reduce(const P &pipe, int s, uint32_t base, uint32_t staged,
                                               uint32_t n, Carry &, const Publish &publish) const
    {
        __shared__ uint32_t s_red[TT::kWarps];
        const int tid = threadIdx.x;
        if constexpr (F32) {
            float a = 0.0f;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                uint32_t x[4];
                stage_load4<FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, r * TT::kRowElems + 4 * tid, staged, n, 0u, x);
                a += (__uint_as_float(x[0]) + __uint_as_float(x[1])) +
                     (__uint_as_float(x[2]) + __uint_as_float(x[3]));
            }
            const uint32_t agg = __float_as_uint(block_sum_all<THREADS>(a, reinterpret_cast<float *>(s_red)));
            publish(agg);
            return agg;
        } else {
            uint32_t a = 0u;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                uint32_t x[4];
                stage_load4<FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, r * TT::kRowElems + 4 * tid, staged, n, 0u, x);
                a += x[0] + x[1] + x[2] + x[3];
            }
            const uint32_t agg = block_sum_all<THREADS>(a, s_red);
            publish(agg);
            return agg;
        }
    }

    template <bool FULL, class P>
    __device__ __forceinline__ void finish(const P &pipe, int s, uint32_t tile, uint32_t base,
                                           uint32_t staged, uint32_t n, uint32_t prefix,
                                           uint32_t agg, bool last, const Carry &,
                                           const Loaded &) const
    {
        __shared__ uint32_t s_chunk[TT::kChunks];
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        uint32_t x[ROWS][4];
        uint32_t lane_excl[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            stage_load4<FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, r * TT::kRowElems + 4 * tid, staged, n, 0u, x[r]);
            const uint32_t v = x[r][0] + x[r][1] + x[r][2] + x[r][3];
            uint32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += y;
            }
            lane_excl[r] = incl - v;
            if (lane == 31) s_chunk[r * TT::kWarps + warp] = incl;
        }
        __syncthreads();
        if (warp == 0) scan_chunks_warp0<TT>(s_chunk);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            uint32_t v = prefix + s_chunk[r * TT::kWarps + warp] + lane_excl[r];
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (INCL) v += x[r][q];   // inclusive: the element itself counts
                o[q] = v;
                if (!INCL) v += x[r][q];
            }
            store4<OUT_VEC && !FULL>(out, base + r * TT::kRowElems + 4 * tid, n, o, FULL && OUT_VEC);
        }
        if (tid == 0 && total != nullptr && last) *total = prefix + agg;
        (void)tile;
    }

    // float32: hi + lo is the tile's exclusive prefix, a float pair carrying
    // about 48 significant bits; each vector's prefix is hi + (lo + its
    // offset inside the tile), rounded once, and each output adds the sum of
    // the vector's elements before it.
    template <bool FULL, class P>
    __device__ __forceinline__ void finish_f32(const P &pipe, int s, uint32_t base, uint32_t staged,
                                               uint32_t n, float hi, float lo, bool last,
                                               float inclusive, const Carry &, const Loaded &) const
    {
        __shared__ float s_chunk[TT::kChunks];
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        uint32_t x[ROWS][4];
        float lane_excl[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            stage_load4<FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, r * TT::kRowElems + 4 * tid, staged, n, 0u, x[r]);
            const float v = (__uint_as_float(x[r][0]) + __uint_as_float(x[r][1])) +
                            (__uint_as_float(x[r][2]) + __uint_as_float(x[r][3]));
            float incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += y;
            }
            const float ex = __shfl_up_sync(kFullMask, incl, 1);
            lane_excl[r] = (lane == 0) ? 0.0f : ex;
            if (lane == 31) s_chunk[r * TT::kWarps + warp] = incl;
        }
        __syncthreads();
        if (warp == 0) scan_chunks_warp0<TT>(s_chunk);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            // the vector's exclusive prefix, once per vector; then each
            // output is that plus the sum inside the vector (one add)
            const float vbase = hi + (lo + (s_chunk[r * TT::kWarps + warp] + lane_excl[r]));
            const float a0 = __uint_as_float(x[r][0]), a1 = __uint_as_float(x[r][1]);
            const float a2 = __uint_as_float(x[r][2]), a3 = __uint_as_float(x[r][3]);
            const float s1 = a0 + a1, s2 = s1 + a2;
            uint32_t o[4];
            if (INCL) {
                o[0] = __float_as_uint(vbase + a0);
                o[1] = __float_as_uint(vbase + s1);
                o[2] = __float_as_uint(vbase + s2);
                o[3] = __float_as_uint(vbase + (s2 + a3));
            } else {
                o[0] = __float_as_uint(vbase);
                o[1] = __float_as_uint(vbase + a0);
                o[2] = __float_as_uint(vbase + s1);
                o[3] = __float_as_uint(vbase + s2);
            }
            store4<OUT_VEC && !FULL>(out, base + r * TT::kRowElems + 4 * tid, n, o, FULL && OUT_VEC);
        }
        if (tid == 0 && total != nullptr && last) *total = __float_as_uint(inclusive);
    }
};

// Predicate masks of one staged tile: bit q of mask[r] says element q of
// the thread's vector r is kept (and lies below n).
template <class TT, bool FULL, bool SH, class Pred>
__device__ __forceinline__ void tile_masks(const uint32_t *sbuf, const uint32_t *gin, uint32_t base,
                                           uint32_t staged, uint32_t n, const Pred &pred,
                                           uint32_t (&mask)[TT::kRows])
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r) {
        const uint32_t li = r * TT::kRowElems + 4 * tid;
        uint32_t x[4];
        stage_load4<FULL, SH>(sbuf, gin, base, li, staged, n, 0u, x);
        uint32_t m = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) m |= uint32_t((FULL || base + li + q < n) && pred(x[q])) << q;
        mask[r] = m;
    }
}

// Reduction of a predicate tile: masks, in-tile ranks and the keep count.
// base[r] = survivors of the tile before this thread's vector r.
template <class TT, bool FULL, bool SH, class Pred, class OnTotal>
__device__ __forceinline__ uint32_t rank_tile(const uint32_t *sbuf, const uint32_t *gin,
                                              uint32_t base, uint32_t staged, uint32_t n,
                                              const Pred &pred, uint32_t (&mask)[TT::kRows],
                                              uint32_t (&rbase)[TT::kRows], const OnTotal &on_total)
{
    __shared__ uint32_t s_chunk[TT::kChunks];
    tile_masks<TT, FULL, SH>(sbuf, gin, base, staged, n, pred, mask);
    uint32_t lane_excl[TT::kRows];
    rank_masks<TT>(mask, lane_excl, s_chunk);
    __syncthreads();
    uint32_t off[TT::kRows], kept;
    chunk_offsets<TT>(s_chunk, off, kept, on_total);
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r) rbase[r] = off[r] + lane_excl[r];
    return kept;
}

// Output placement of a select-if: survivors go to out[obase + rank], and a
// tile whose run would end past cap records GC_ERR_DEVICE_CHECK and stores
// nothing (obase = null, read as 0, and cap = n for the plain entry point).
struct SelectPlacement {
    const uint64_t *obase;
    uint64_t cap;
};

// Stable select-if.  The tile's survivors are compacted in place inside its
// own stage buffer (every element was read into registers before the barrier
// that precedes the first write, and a survivor's rank never exceeds its
// index), shifted so that shared and global addresses agree modulo 16 bytes,
// then written as one contiguous run with 128-bit stores.
template <int THREADS, int ROWS, class Pred, bool VEC, bool PLACED = false, bool SH = false>
struct SelectOp {
    using TT = Tile<THREADS, ROWS>;
    static constexpr uint32_t kTileElems = TT::kElems;
    static constexpr bool kF32 = false;
    template <int STAGES>
    using PipeT = Pipe<kTileElems * 4u, STAGES, 1>;

    const uint32_t *srcs[1];
    uint32_t *out;
    uint32_t *count;
    Pred pred;
    SelectPlacement place;
    uint8_t *ws;  // the error word of a refused run

    struct Carry {
        uint32_t mask[ROWS];
        uint32_t base[ROWS];
    };
    __device__ __forceinline__ void seed(uint32_t &, float &, float &) const {}
    // The tile is read into registers before the window barrier, which then
    // also orders those reads before the in-place compaction's writes.
    static constexpr bool kPreload = true;
    struct Loaded {
        uint32_t x[ROWS][4];
    };

    template <bool FULL, class P, class Publish>
    __device__ __forceinline__ uint32_t reduce(const P &pipe, int s, uint32_t base, uint32_t staged,
                                               uint32_t n, Carry &c, const Publish &publish) const
    {
        // The count goes out before the per-row ranks are derived.
        return rank_tile<TT, FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, staged, n, pred, c.mask, c.base, publish);
    }

    // A tile with fewer survivors than this skips the in-place compaction:
    // each thread stores its few survivors straight from the stage buffer.
    static constexpr uint32_t kSparse = TT::kElems / 16;

    template <bool FULL, class P>
    __device__ __forceinline__ void load(const P &pipe, int s, uint32_t base, uint32_t staged,
                                         uint32_t n, uint32_t kept, Loaded &ld) const
    {
        if (kept >= kSparse) tile_vectors<TT, FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, staged, n, ld.x);
    }

    template <bool FULL, class P>
    __device__ __forceinline__ void finish(const P &pipe, int s, uint32_t tile, uint32_t base,
                                           uint32_t staged, uint32_t n, uint32_t before,
                                           uint32_t kept, bool last, const Carry &c,
                                           const Loaded &ld) const
    {
        uint32_t *buf = pipe.buf(s);          // written: in-place compaction
        const uint32_t *rbuf = stage_rd<SH>(pipe, s);  // read: element j at rbuf[j]
        if (threadIdx.x == 0 && last) *count = before + kept;
        uint32_t *o = out;
        uint32_t d0 = before;  // index into o
        if constexpr (PLACED) {
            // placed output: out[obase + before + rank], refused past cap
            const uint64_t ob = __ldg(place.obase);
            if (ob + before + kept > place.cap) {
                if (threadIdx.x == 0) record_error(ws, kDeviceCheckCode, tile);
                return;
            }
            o = out + (ob & ~3ull);
            d0 = uint32_t(ob & 3ull) + before;
        }
        if (kept < kSparse) {
            // Survivor q of vector r goes to before + base[r] + (survivors of
            // the vector before it); no shared-memory writes, so no barrier.
            // The thread's survivors in one loop over the set bits of its
            // eight masks side by side (bit 4r + q), so a warp runs as many
            // iterations as its busiest lane has survivors (a loop per row
            // ran up to eight dependent load-store chains: 67.0 -> 63.0 us at
            // 1% kept and 2^26).
            static_assert(ROWS <= 8, "eight 4-bit masks to a word");
            uint32_t all = 0u;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) all |= c.mask[r] << (4 * r);
            uint32_t left = all;
            while (left != 0u) {
                const uint32_t b = uint32_t(__ffs(left) - 1);
                left &= left - 1u;
                const uint32_t r = b >> 2, q = b & 3u;
                uint32_t rbase = c.base[0];
#pragma unroll
                for (int rr = 1; rr < ROWS; ++rr)
                    if (r == uint32_t(rr)) rbase = c.base[rr];
                const uint32_t pos = d0 + rbase + uint32_t(__popc((all >> (4u * r)) & ((1u << q) - 1u)));
                const uint32_t li = r * TT::kRowElems + 4u * threadIdx.x;
                const uint32_t x = (FULL || li + 4u <= staged) ? rbuf[li + q] : srcs[0][base + li + q];
                __stcs(o + pos, x);
            }
            return;
        }
        const uint32_t shift = VEC ? (d0 & 3u) : 0u;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            uint32_t pos = shift + c.base[r];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if ((c.mask[r] >> q) & 1u) buf[pos++] = ld.x[r][q];
        }
        if (VEC && kept >= kBulkMinRun) {
            fence_proxy_async_smem();
            __syncthreads();
            store_run_bulk<THREADS>(o, d0, buf, shift, kept, 0);
        } else {
            __syncthreads();
            store_run<THREADS, VEC>(o, d0, buf, shift, kept);
        }
    }
};

// Predicate masks of one staged tile: bit q of mask[r] says element q of
// thread's vector r is kept (and lies below n).
template <class TT, bool FULL, bool SH, class Pred>
__device__ __forceinline__ void tile_masks_x(const uint32_t *sbuf, const uint32_t *gin, uint32_t base,
                                           uint32_t staged, uint32_t n, const Pred &pred,
                                           uint32_t (&x)[TT::kRows][4], uint32_t (&mask)[TT::kRows])
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r) {
        const uint32_t li = r * TT::kRowElems + 4 * tid;
        stage_load4<FULL, SH>(sbuf, gin, base, li, staged, n, 0u, x[r]);
        uint32_t m = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) m |= uint32_t((FULL || base + li + q < n) && pred(x[r][q])) << q;
        mask[r] = m;
    }
}

// Keep count of one staged tile, to every thread; the masks it finds are
// left in `mask` for the tile's finish a round later.
template <class TT, bool FULL, bool SH, class Pred>
__device__ __forceinline__ uint32_t tile_count(const uint32_t *sbuf, const uint32_t *gin,
                                               uint32_t base, uint32_t staged, uint32_t n,
                                               const Pred &pred, uint32_t *s_red,
                                               uint32_t (&mask)[TT::kRows])
{
    uint32_t x[TT::kRows][4];
    tile_masks_x<TT, FULL, SH>(sbuf, gin, base, staged, n, pred, x, mask);
    uint32_t c = 0u;
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r) c += __popc(mask[r]);
    return block_sum_all<TT::kThreads>(c, s_red);
}

// Stable partition (and the radix one-bit split, with payloads): kept
// elements go to [before, before + kept) and rejected ones to
// T + (base - before) onwards, the i - rank[i] addressing of "compaction.cu
// -- Day 33" (scatterPartition), with T the total kept from the pre-pass.
// Both runs are compacted in place in the stage buffer(s) and written with
// 128-bit stores.
template <int THREADS, int ROWS, class Pred, bool VEC, bool VALS, bool PLACED = false, bool SH = false>
struct PartitionOp {
    using TT = Tile<THREADS, ROWS>;
    static constexpr uint32_t kTileElems = TT::kElems;
    static constexpr bool kF32 = false;
    template <int STAGES>
    using PipeT = Pipe<kTileElems * 4u, STAGES, VALS ? 2 : 1>;

    const uint32_t *srcs[VALS ? 2 : 1];
    uint32_t *keys_out;
    uint32_t *vals_out;
    const uint32_t *true_total;  // written by the pre-pass kernel
    uint8_t *ws;
    Pred pred;
    // Placed output (a shard of a larger partition): kept elements go to
    // out[offsets[0] + rank], rejected ones to out[offsets[1] + i - rank],
    // runs checked against capacity, and the last tile writes the tile
    // total to count_out.  offsets == nullptr: the plain partition, kept
    // from 0 and rejected from *true_total.
    const uint64_t *offsets;
    uint64_t capacity;
    uint32_t *count_out;

    struct Carry {
        uint32_t mask[ROWS];
    };
    __device__ __forceinline__ void seed(uint32_t &, float &, float &) const {}
    static constexpr bool kPreload = false;
    struct Loaded {};

    template <bool FULL, class P>
    __device__ __forceinline__ void load(const P &, int, uint32_t, uint32_t, uint32_t, uint32_t,
                                         Loaded &) const {}

    template <bool FULL, class P, class Publish>
    __device__ __forceinline__ uint32_t reduce(const P &pipe, int s, uint32_t base, uint32_t staged,
                                               uint32_t n, Carry &c, const Publish &publish) const
    {
        __shared__ uint32_t s_red[TT::kWarps];
        const uint32_t agg = tile_count<TT, FULL, SH>(stage_rd<SH>(pipe, s), srcs[0], base, staged, n, pred, s_red, c.mask);
        publish(agg);
        return agg;
    }

    template <bool FULL, class P>
    __device__ __forceinline__ void finish(const P &pipe, int s, uint32_t tile, uint32_t base,
                                           uint32_t staged, uint32_t n, uint32_t before,
                                           uint32_t kept, bool last, const Carry &c,
                                           const Loaded &) const
    {
        __shared__ uint32_t s_chunk[TT::kChunks];
        const int tid = threadIdx.x, warp = tid >> 5;
        uint32_t *kbuf = pipe.buf(s, 0);  // written: in-place compaction of both runs
        uint32_t *vbuf = pipe.buf(s, VALS ? 1 : 0);
        uint32_t x[ROWS][4], lane_excl[ROWS];
        uint32_t v[VALS ? ROWS : 1][4];
        tile_vectors<TT, FULL, SH>(stage_rd<SH>(pipe, s, 0), srcs[0], base, staged, n, x);
        const uint32_t (&mask)[ROWS] = c.mask;
        if (VALS) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                stage_load4<FULL, SH>(stage_rd<SH>(pipe, s, VALS ? 1 : 0), srcs[VALS ? 1 : 0], base, r * TT::kRowElems + 4 * tid, staged,
                                  n, 0u, v[VALS ? r : 0]);
        }
        rank_masks<TT>(mask, lane_excl, s_chunk);
        uint64_t kbase = 0u, rbase, cap = n;
        if constexpr (PLACED) {
            kbase = offsets[0];
            rbase = offsets[1];
            cap = capacity;
        } else {
            rbase = *true_total;
        }
        __syncthreads();
        if (warp == 0) scan_chunks_warp0<TT>(s_chunk);
        __syncthreads();

        const uint32_t valid = min(kTileElems, n - base);
        uint32_t rejected = valid - kept;
        uint32_t kept_len = kept;
        if (PLACED && tid == 0 && last) *count_out = before + kept;
        // Both runs must lie inside the output, which holds when T (or the
        // placed offsets) are right; a wrong value (a workspace corrupted
        // between the two kernels, a bad offset) is recorded and the stores
        // are skipped.
        uint32_t *kout_k = keys_out, *kout_r = keys_out, *vout_k = vals_out, *vout_r = vals_out;
        uint32_t dst_kept, dst_rej;
        if constexpr (PLACED) {
            const uint64_t gk = kbase + before, gr = rbase + (base - before);
            if (gr + rejected > cap || gk + kept > cap) {
                if (tid == 0) record_error(ws, kDeviceCheckCode, tile);
                kept_len = 0u;
                rejected = 0u;
            }
            dst_kept = uint32_t(gk & 3u);
            dst_rej = uint32_t(gr & 3u);
            kout_k = keys_out + (gk & ~3ull);
            kout_r = keys_out + (gr & ~3ull);
            if (VALS) {
                vout_k = vals_out + (gk & ~3ull);
                vout_r = vals_out + (gr & ~3ull);
            }
        } else {
            const uint32_t T = uint32_t(rbase);
            dst_kept = before;
            dst_rej = T + (base - before);
            if (uint64_t(dst_rej) + rejected > cap || uint64_t(dst_kept) + kept > T) {
                if (tid == 0) record_error(ws, kDeviceCheckCode, tile);
                kept_len = 0u;
                rejected = 0u;
            }
        }
        const uint32_t sh_kept = VEC ? (dst_kept & 3u) : 0u;
        const uint32_t rej_region = (sh_kept + kept + 3u) & ~3u;
        const uint32_t sh_rej = rej_region + (VEC ? (dst_rej & 3u) : 0u);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const uint32_t local0 = r * TT::kRowElems + 4 * tid;
            uint32_t ranked = s_chunk[r * TT::kWarps + warp] + lane_excl[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t local = local0 + q;
                if (FULL || base + local < n) {
                    const bool keep = (mask[r] >> q) & 1u;
                    const uint32_t slot = keep ? sh_kept + ranked : sh_rej + (local - ranked);
                    kbuf[slot] = x[r][q];
                    if (VALS) vbuf[slot] = v[VALS ? r : 0][q];
                    ranked += keep ? 1u : 0u;
                }
            }
        }
        if (VEC && valid >= kBulkMinRun) {
            // The runs leave by bulk copies from the stage buffer(s).
            fence_proxy_async_smem();
            __syncthreads();
            store_run_bulk<THREADS>(kout_k, dst_kept, kbuf, sh_kept, kept_len, 0);
            store_run_bulk<THREADS>(kout_r, dst_rej, kbuf, sh_rej, rejected, 1);
            if (VALS) {
                store_run_bulk<THREADS>(vout_k, dst_kept, vbuf, sh_kept, kept_len, 2);
                store_run_bulk<THREADS>(vout_r, dst_rej, vbuf, sh_rej, rejected, 3);
            }
        } else {
            __syncthreads();
            store_run<THREADS, VEC>(kout_k, dst_kept, kbuf, sh_kept, kept_len);
            store_run<THREADS, VEC>(kout_r, dst_rej, kbuf, sh_rej, rejected);
            if (VALS) {
                store_run<THREADS, VEC>(vout_k, dst_kept, vbuf, sh_kept, kept_len);
                store_run<THREADS, VEC>(vout_r, dst_rej, vbuf, sh_rej, rejected);
            }
        }
        (void)last;
    }
};

}  // namespace gcd
