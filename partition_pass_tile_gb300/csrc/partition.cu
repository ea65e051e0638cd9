// partition.cu -- stable two-way partition, the one-bit split and the LSD
// radix sort built from it.
//
// "compaction.cu -- Day 33" (partitionCpu, scatterPartition): rank[i], the
// number of kept elements before i, addresses the kept half directly, and
// i - rank[i] is the number of rejected elements before i, so one scan
// addresses both halves; the rejected half starts at T, the total kept, which
// must be known before anything is scattered.  T therefore comes from a count
// pre-pass (count_kernel: one read of the input, a block reduction, one
// atomic per CTA, and the last CTA to finish publishes the total), and the
// main pass is the single-pass tile kernel of select.cu with two output runs
// per tile instead of one.
//
// The radix sort ("CIS 565 Project 2: Stream Compaction", radix sort built
// on scan) is that partition with the predicate "bit b clear", applied to
// (key, payload) pairs once per bit from the lowest.  The number of keys with
// bit b clear does not change when keys are permuted, so one histogram pass
// over the input gives T for all 32 splits.
#include "gc_device.cuh"
#include "gc_internal.h"
#include "gc_launch.cuh"

namespace {

using namespace gcd;

constexpr int kPad = 12;  // shared staging slack: two runs, each shifted by up to 3

template <class Pred, int THREADS, int ROWS, bool VEC, bool VALS, bool LB>
__global__ void __launch_bounds__(THREADS)
partition_kernel(const uint32_t *__restrict__ keys_in, const uint32_t *__restrict__ vals_in,
                 uint32_t *__restrict__ keys_out, uint32_t *__restrict__ vals_out, uint32_t n,
                 uint32_t num_tiles, const uint32_t *true_total, Pred pred, uint8_t *ws,
                 uint64_t timeout_ns, const uint64_t *offsets, uint64_t capacity,
                 uint32_t *count_out)
{
    using TT = Tile<THREADS, ROWS>;
    __shared__ uint32_t s_tile;
    __shared__ uint32_t s_chunk[TT::kChunks];
    __shared__ PrefixSmem s_ps;
    __shared__ uint32_t s_total;
    __shared__ __align__(16) uint32_t s_keys[TT::kElems + kPad];
    __shared__ __align__(16) uint32_t s_vals[VALS ? TT::kElems + kPad : 4];

    const uint32_t tile = claim_tile(ws, &s_tile);
    if (tile >= num_tiles) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t base = tile * uint32_t(TT::kElems);

    uint32_t x[ROWS][4];
    uint32_t v[VALS ? ROWS : 1][4];
    uint32_t mask[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const uint32_t idx = base + r * TT::kRowElems + 4 * tid;
        load4<VEC>(keys_in, idx, n, 0u, x[r]);
        if (VALS) load4<VEC>(vals_in, idx, n, 0u, v[VALS ? r : 0]);
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) m |= uint32_t(idx + k < n && pred(x[r][k])) << k;
        mask[r] = m;
    }

    uint32_t lane_excl[ROWS];
    rank_masks<TT>(mask, lane_excl, s_chunk);
    __syncthreads();

    if (tid == 0 && offsets == nullptr) s_total = *true_total;
    uint32_t before, kept;
    resolve_prefix_u32<TT, LB>(s_chunk, tile, ws, timeout_ns, s_ps, before, kept);
    if (tid == 0 && count_out != nullptr && tile == num_tiles - 1) *count_out = before + kept;
    const uint32_t valid = min(uint32_t(TT::kElems), n - base);
    const uint32_t rejected = valid - kept;
    // Kept elements from kbase + rank[i], rejected ones from rbase + i - rank[i]
    // (rbase = T for the plain partition, the placed offsets otherwise).
    const uint64_t kbase = offsets != nullptr ? offsets[0] : 0u;
    const uint64_t rbase = offsets != nullptr ? offsets[1] : s_total;
    const uint64_t cap = offsets != nullptr ? capacity : n;
    const uint64_t gk = kbase + before, gr = rbase + (base - before);
    // Both runs must lie inside the output: true only if T (or the offsets)
    // are right.  A wrong value (a workspace corrupted between the kernels) is
    // recorded and the stores are skipped instead of landing out of range.
    if (gr + rejected > cap || gk + kept > cap || (offsets == nullptr && gk + kept > rbase)) {
        if (tid == 0) record_error(ws, kDeviceCheckCode, tile);
        return;
    }
    const uint32_t dst_kept = uint32_t(gk & 3u), dst_rej = uint32_t(gr & 3u);
    uint32_t *const kout_k = keys_out + (gk & ~3ull), *const kout_r = keys_out + (gr & ~3ull);
    uint32_t *const vout_k = VALS ? vals_out + (gk & ~3ull) : nullptr;
    uint32_t *const vout_r = VALS ? vals_out + (gr & ~3ull) : nullptr;
    const uint32_t sh_kept = VEC ? (dst_kept & 3u) : 0u;
    const uint32_t rej_region = (sh_kept + kept + 3u) & ~3u;
    const uint32_t sh_rej = rej_region + (VEC ? (dst_rej & 3u) : 0u);

#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const uint32_t local0 = r * TT::kRowElems + 4 * tid;
        uint32_t ranked = s_chunk[r * TT::kWarps + warp] + lane_excl[r];  // kept before this item
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t local = local0 + k;
            if (base + local < n) {
                const uint32_t slot = ((mask[r] >> k) & 1u) ? sh_kept + ranked
                                                            : sh_rej + (local - ranked);
                s_keys[slot] = x[r][k];
                if (VALS) s_vals[slot] = v[VALS ? r : 0][k];
                ranked += (mask[r] >> k) & 1u;
            }
        }
    }
    __syncthreads();
    store_run<THREADS, VEC>(kout_k, dst_kept, s_keys, sh_kept, kept);
    store_run<THREADS, VEC>(kout_r, dst_rej, s_keys, sh_rej, rejected);
    if (VALS) {
        store_run<THREADS, VEC>(vout_k, dst_kept, s_vals, sh_kept, kept);
        store_run<THREADS, VEC>(vout_r, dst_rej, s_vals, sh_rej, rejected);
    }
}

// Sum of one uint32 over the CTA, returned to thread 0.
template <int THREADS>
__device__ __forceinline__ uint32_t block_sum(uint32_t c, uint32_t *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    c = warp_sum(c);
    if (lane == 0) s_warp[warp] = c;
    __syncthreads();
    uint32_t t = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < THREADS / 32; ++w) t += s_warp[w];
    return t;
}

// Count pre-pass of the partition: how many elements the predicate keeps.
// Each CTA adds its count to an accumulator in the workspace header; the CTA
// that finishes last (by a ticket counter) takes the sum, resets both words
// for the next call, and publishes the total.
template <class Pred, int THREADS, bool VEC>
__global__ void __launch_bounds__(THREADS)
count_kernel(const uint32_t *__restrict__ in, uint32_t n, Pred pred, uint8_t *ws,
             uint32_t *count_out)
{
    __shared__ uint32_t s_warp[THREADS / 32];
    constexpr uint32_t kUnroll = 4;
    const uint32_t nvec = (n + 3u) / 4u;
    const uint32_t stride = gridDim.x * THREADS;
    uint32_t c = 0;
    for (uint32_t v0 = blockIdx.x * THREADS + threadIdx.x; v0 < nvec; v0 += stride * kUnroll) {
        uint32_t x[kUnroll][4];
#pragma unroll
        for (uint32_t u = 0; u < kUnroll; ++u) {
            const uint32_t v = v0 + u * stride;
            if (v < nvec) load4<VEC>(in, 4u * v, n, 0u, x[u]);
        }
#pragma unroll
        for (uint32_t u = 0; u < kUnroll; ++u) {
            const uint32_t v = v0 + u * stride;
            if (v < nvec) {
#pragma unroll
                for (int k = 0; k < 4; ++k) c += uint32_t(4u * v + k < n && pred(x[u][k]));
            }
        }
    }
    const uint32_t total = block_sum<THREADS>(c, s_warp);
    if (threadIdx.x == 0) {
        atomicAdd(hdr_u32(ws, kHdrCountAcc), total);
        __threadfence();
        const uint32_t ticket = atomicAdd(hdr_u32(ws, kHdrReduceCtr), 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const uint32_t all = atomicExch(hdr_u32(ws, kHdrCountAcc), 0u);
            atomicExch(hdr_u32(ws, kHdrReduceCtr), 0u);
            *hdr_u32(ws, kHdrCountTrue) = all;
            *count_out = all;
        }
    }
}

// Carry-save adder: l + 2h = a + b + c, bit by bit.
__device__ __forceinline__ void csa(uint32_t &h, uint32_t &l, uint32_t a, uint32_t b, uint32_t c)
{
    const uint32_t u = a ^ b;
    h = (a & b) | (u & c);
    l = u ^ c;
}

// Radix histogram: for every bit b, how many keys have it set.  Keys are
// counted eight at a time in bit-sliced form (the carry-save tree of the
// Harley-Seal population count): seven adders fold eight keys into the
// running ones, twos and fours words and one "eights" word, whose bit b says
// that eight more keys have bit b set.  Only that word is spread into
// per-bit counters, eight bits at a time in byte lanes ((w >> j) &
// 0x01010101 holds bits j, j+8, j+16, j+24 as four byte-wide 0/1 values),
// spilled into 32 wide counters every 255 groups before a byte can
// overflow; the ones, twos and fours words are added in at the end.
// Reduced across the warp with a butterfly that leaves bit b's total in
// lane b, then across the CTA and the grid as in count_kernel; the last CTA
// stores n - ones as the clear-bit count.
// KEYED counts the bits of the order-preserving key x ^ (signfill(x) & neg)
// ^ flip instead of x (see PredKeyBitClear); the padding past n in the last
// vector loads as 0, whose key is flip, and the last CTA takes those bits
// back out.
template <int THREADS, bool VEC, bool KEYED>
__global__ void __launch_bounds__(THREADS)
bit_histogram_kernel(const uint32_t *__restrict__ keys, uint32_t n, uint8_t *ws, uint32_t neg,
                     uint32_t flip)
{
    __shared__ uint32_t s_ones[32];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) s_ones[threadIdx.x] = 0u;
    __syncthreads();

    uint32_t ones[32];
#pragma unroll
    for (int b = 0; b < 32; ++b) ones[b] = 0u;
    uint32_t acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0u;
    uint32_t in_acc = 0;  // eights words added to acc since the last spill (<= 255)
    uint32_t w1 = 0u, w2 = 0u, w4 = 0u;  // bit-sliced counts 0..7 per bit position

    const uint32_t nvec = (n + 3u) / 4u;
    const uint32_t stride = gridDim.x * THREADS;
    for (uint32_t v = blockIdx.x * THREADS + threadIdx.x; v < nvec; v += 2u * stride) {
        uint32_t x[4], y[4];
        load4<VEC>(keys, 4u * v, n, 0u, x);  // padding keys are 0: no bits set
        const bool have_y = v + stride < nvec;
        if (have_y)
            load4<VEC>(keys, 4u * (v + stride), n, 0u, y);
        else
            y[0] = y[1] = y[2] = y[3] = 0u;
        if (KEYED) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[k] ^= (uint32_t(int32_t(x[k]) >> 31) & neg) ^ flip;
                y[k] = have_y ? y[k] ^ ((uint32_t(int32_t(y[k]) >> 31) & neg) ^ flip) : 0u;
            }
        }
        uint32_t t2a, t2b, t4a, t4b, w8;
        csa(t2a, w1, w1, x[0], x[1]);
        csa(t2b, w1, w1, x[2], x[3]);
        csa(t4a, w2, w2, t2a, t2b);
        csa(t2a, w1, w1, y[0], y[1]);
        csa(t2b, w1, w1, y[2], y[3]);
        csa(t4b, w2, w2, t2a, t2b);
        csa(w8, w4, w4, t4a, t4b);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += (w8 >> j) & 0x01010101u;
        if (++in_acc == 255u) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int q = 0; q < 4; ++q) ones[8 * q + j] += 8u * ((acc[j] >> (8 * q)) & 0xffu);
                acc[j] = 0u;
            }
            in_acc = 0;
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) ones[8 * q + j] += 8u * ((acc[j] >> (8 * q)) & 0xffu);
#pragma unroll
    for (int b = 0; b < 32; ++b)
        ones[b] += ((w1 >> b) & 1u) + 2u * ((w2 >> b) & 1u) + 4u * ((w4 >> b) & 1u);

    // Butterfly reduce-scatter: after the step with offset o each lane keeps
    // the half of its array selected by (lane & o); at the end lane l holds
    // the warp's total for bit l in ones[0].
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const uint32_t send = upper ? ones[i] : ones[i + o];
            const uint32_t keep = upper ? ones[i + o] : ones[i];
            ones[i] = keep + __shfl_xor_sync(kFullMask, send, o);
        }
    }
    atomicAdd(&s_ones[lane], ones[0]);
    __syncthreads();
    if (threadIdx.x < 32) {
        atomicAdd(hdr_u32(ws, kHdrBitAcc + 4u * threadIdx.x), s_ones[threadIdx.x]);
        __threadfence();  // this thread's add is visible before the ticket below
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t ticket = atomicAdd(hdr_u32(ws, kHdrReduceCtr), 1u);
        s_ones[0] = (ticket == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_ones[0] != 0u && threadIdx.x < 32) {
        __threadfence();
        uint32_t total_ones = atomicExch(hdr_u32(ws, kHdrBitAcc + 4u * threadIdx.x), 0u);
        if (KEYED) total_ones -= (4u * ((n + 3u) / 4u) - n) * ((flip >> threadIdx.x) & 1u);
        *hdr_u32(ws, kHdrBitZeros + 4u * threadIdx.x) = n - total_ones;
        if (threadIdx.x == 0) atomicExch(hdr_u32(ws, kHdrReduceCtr), 0u);
    }
}

int reduce_grid(uint32_t n, int threads)
{
    const size_t want = gch::ceil_div(gch::ceil_div(n, 4), size_t(threads));
    const size_t cap = size_t(gch::sm_count()) * 8;
    return int(want < cap ? (want > 0 ? want : 1) : cap);
}

// Where a partition pass puts its runs: the plain partition (offsets null:
// kept from 0, rejected from the device-side T) or a placed shard.
struct PartPlace {
    const uint64_t *offsets = nullptr;
    uint64_t capacity = 0;
    uint32_t *count_out = nullptr;
};

template <int PT, int PR, int PS, class Pred, bool VALS>
cudaError_t run_partition_pipe(const uint32_t *kin, const uint32_t *vin, uint32_t *kout,
                               uint32_t *vout, uint32_t n, const uint32_t *true_total, Pred pred,
                               uint8_t *ws, cudaStream_t s, const gch::LaunchOpts &o,
                               const PartPlace &pl)
{
    const bool vec = gch::aligned16(kout) && (!VALS || gch::aligned16(vout));
    auto fill = [&](auto &op) {
        op.srcs[0] = kin;
        if constexpr (VALS) op.srcs[VALS ? 1 : 0] = vin;
        op.keys_out = kout;
        op.vals_out = vout;
        op.true_total = true_total;
        op.ws = ws;
        op.pred = pred;
        op.offsets = pl.offsets;
        op.capacity = pl.capacity;
        op.count_out = pl.count_out;
    };
    auto go = [&](auto op) {
        fill(op);
        return gcd::launch_pipeline<PT, PS>(op, n, ws, s, o);
    };
    // The placed form (a shard of a larger partition) is its own
    // instantiation, so the plain partition and the radix splits keep their
    // 32-bit addressing.
    // Inputs that are not 16-byte aligned are staged shifted, with the runs
    // stored element by element.
    const bool shifted = !gch::aligned16(kin) || (VALS && !gch::aligned16(vin));
    if (pl.offsets != nullptr) {
        if constexpr (!VALS) {
            if (shifted) return go(gcd::PartitionOp<PT, PR, Pred, false, VALS, true, true>{});
            if (vec) return go(gcd::PartitionOp<PT, PR, Pred, true, VALS, true>{});
            return go(gcd::PartitionOp<PT, PR, Pred, false, VALS, true>{});
        }
        return cudaErrorNotSupported;
    }
    if (shifted) return go(gcd::PartitionOp<PT, PR, Pred, false, VALS, false, true>{});
    if (vec) return go(gcd::PartitionOp<PT, PR, Pred, true, VALS, false>{});
    return go(gcd::PartitionOp<PT, PR, Pred, false, VALS, false>{});
}

// *piped (optional) says whether the persistent kernel ran; the fallback
// kernels clear their own status words (region 0) with a memset and ignore
// o's status plan.
template <class Pred, bool VALS>
cudaError_t run_partition_pass(const uint32_t *kin, const uint32_t *vin, uint32_t *kout,
                               uint32_t *vout, uint32_t n, const uint32_t *true_total, Pred pred,
                               uint8_t *ws, cudaStream_t s, const gch::LaunchOpts &o, bool split,
                               bool *piped = nullptr, const PartPlace &pl = PartPlace{})
{
    if (piped != nullptr) *piped = false;
    if (!o.skip_first_tile && !gch::force_fallback()) {
        cudaError_t e;
        if (split)
            e = run_partition_pipe<gch::kSplitPipeThreads, gch::kSplitPipeRows, gch::kSplitPipeStages,
                                   Pred, VALS>(kin, vin, kout, vout, n, true_total, pred, ws, s, o, pl);
        else
            e = run_partition_pipe<gch::kPartPipeThreads, gch::kPartPipeRows, gch::kPartPipeStages,
                                   Pred, VALS>(kin, vin, kout, vout, n, true_total, pred, ws, s, o, pl);
        if (e == cudaSuccess) {
            if (piped != nullptr) *piped = true;
            return e;
        }
        (void)cudaGetLastError();  // cooperative grid refused: one tile per CTA instead
    }
    constexpr int PT = gch::kPartThreads, PR = gch::kPartRows;
    constexpr int ST = gch::kSplitThreads, SR = gch::kSplitRows;
    const uint32_t tile = split ? gch::tile_elems(ST, SR) : gch::tile_elems(PT, PR);
    const uint32_t tiles = uint32_t(gch::ceil_div(n, tile));
    cudaError_t e = gch::reset_tiles(ws, tiles, s, o.skip_first_tile);
    if (e != cudaSuccess) return e;
    const uint32_t grid = o.skip_first_tile ? tiles - 1 : tiles;
    if (grid == 0) return cudaSuccess;
    const bool vec = gch::aligned16(kin) && gch::aligned16(kout) &&
                     (!VALS || (gch::aligned16(vin) && gch::aligned16(vout)));
    if (split) {
        if (vec)
            partition_kernel<Pred, ST, SR, true, VALS, gch::kCtaLookback><<<grid, ST, 0, s>>>(
                kin, vin, kout, vout, n, tiles, true_total, pred, ws, o.timeout_ns, pl.offsets, pl.capacity, pl.count_out);
        else
            partition_kernel<Pred, ST, SR, false, VALS, gch::kCtaLookback><<<grid, ST, 0, s>>>(
                kin, vin, kout, vout, n, tiles, true_total, pred, ws, o.timeout_ns, pl.offsets, pl.capacity, pl.count_out);
    } else {
        if (vec)
            partition_kernel<Pred, PT, PR, true, VALS, gch::kCtaLookback><<<grid, PT, 0, s>>>(
                kin, vin, kout, vout, n, tiles, true_total, pred, ws, o.timeout_ns, pl.offsets, pl.capacity, pl.count_out);
        else
            partition_kernel<Pred, PT, PR, false, VALS, gch::kCtaLookback><<<grid, PT, 0, s>>>(
                kin, vin, kout, vout, n, tiles, true_total, pred, ws, o.timeout_ns, pl.offsets, pl.capacity, pl.count_out);
    }
    return cudaGetLastError();
}

template <class Pred>
cudaError_t dispatch_partition(const uint32_t *in, uint32_t *out, uint32_t *count_true,
                               uint32_t n, Pred pred, uint8_t *ws, cudaStream_t s,
                               const gch::LaunchOpts &o)
{
    constexpr int RT = gch::kReduceThreads;
    const int grid = reduce_grid(n, RT);
    cudaError_t e0 = gch::clear_accumulators(ws, s);
    if (e0 != cudaSuccess) return e0;
    if (gch::aligned16(in))
        count_kernel<Pred, RT, true><<<grid, RT, 0, s>>>(in, n, pred, ws, count_true);
    else
        count_kernel<Pred, RT, false><<<grid, RT, 0, s>>>(in, n, pred, ws, count_true);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const uint32_t *T = reinterpret_cast<const uint32_t *>(ws + kHdrCountTrue);
    return run_partition_pass<Pred, false>(in, nullptr, out, nullptr, n, T, pred, ws, s, o, false);
}

// A shard of a larger partition: the offsets are known (from the counts of
// every shard), so no pre-pass; one pass writes both runs and the count.
template <class Pred>
cudaError_t dispatch_partition_at(const uint32_t *in, uint32_t *out, uint64_t capacity,
                                  const uint64_t *offsets, uint32_t *count_true, uint32_t n,
                                  Pred pred, uint8_t *ws, cudaStream_t s, const gch::LaunchOpts &o)
{
    PartPlace pl;
    pl.offsets = offsets;
    pl.capacity = capacity;
    pl.count_out = count_true;
    return run_partition_pass<Pred, false>(in, nullptr, out, nullptr, n, nullptr, pred, ws, s, o,
                                           false, nullptr, pl);
}

// Count pre-pass alone (gc_count_if).
template <class Pred>
cudaError_t dispatch_count(const uint32_t *in, uint32_t *count, uint32_t n, Pred pred, uint8_t *ws,
                           cudaStream_t s)
{
    constexpr int RT = gch::kReduceThreads;
    const int grid = reduce_grid(n, RT);
    cudaError_t e0 = gch::clear_accumulators(ws, s);
    if (e0 != cudaSuccess) return e0;
    if (gch::aligned16(in))
        count_kernel<Pred, RT, true><<<grid, RT, 0, s>>>(in, n, pred, ws, count);
    else
        count_kernel<Pred, RT, false><<<grid, RT, 0, s>>>(in, n, pred, ws, count);
    return cudaGetLastError();
}

}  // namespace

namespace gch {

uint32_t partition_tile_elems() { return tile_elems(kPartPipeThreads, kPartPipeRows); }
uint32_t split_tile_elems() { return tile_elems(kSplitPipeThreads, kSplitPipeRows); }

cudaError_t launch_partition(const void *in, void *out, uint32_t *count_true, uint32_t n,
                             gc_dtype dt, gc_pred p, uint8_t *ws, cudaStream_t s,
                             const LaunchOpts &o)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    switch (p) {
    case GC_PRED_NONZERO:
        if (dt == GC_F32) return dispatch_partition(i, u, count_true, n, gcd::PredNonzeroF32{}, ws, s, o);
        return dispatch_partition(i, u, count_true, n, gcd::PredNonzeroInt{}, ws, s, o);
    case GC_PRED_ODD: return dispatch_partition(i, u, count_true, n, gcd::PredOdd{}, ws, s, o);
    default: return dispatch_partition(i, u, count_true, n, gcd::PredEven{}, ws, s, o);
    }
}

cudaError_t launch_partition_at(const void *in, void *out, uint64_t capacity,
                                const uint64_t *offsets, uint32_t *count_true, uint32_t n,
                                gc_dtype dt, gc_pred p, uint8_t *ws, cudaStream_t s,
                                const LaunchOpts &o)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    switch (p) {
    case GC_PRED_NONZERO:
        if (dt == GC_F32)
            return dispatch_partition_at(i, u, capacity, offsets, count_true, n, gcd::PredNonzeroF32{}, ws, s, o);
        return dispatch_partition_at(i, u, capacity, offsets, count_true, n, gcd::PredNonzeroInt{}, ws, s, o);
    case GC_PRED_ODD: return dispatch_partition_at(i, u, capacity, offsets, count_true, n, gcd::PredOdd{}, ws, s, o);
    default: return dispatch_partition_at(i, u, capacity, offsets, count_true, n, gcd::PredEven{}, ws, s, o);
    }
}

cudaError_t launch_count_if(const void *in, uint32_t *count, uint32_t n, gc_dtype dt, gc_pred p,
                            uint8_t *ws, cudaStream_t s)
{
    auto *i = static_cast<const uint32_t *>(in);
    switch (p) {
    case GC_PRED_NONZERO:
        if (dt == GC_F32) return dispatch_count(i, count, n, gcd::PredNonzeroF32{}, ws, s);
        return dispatch_count(i, count, n, gcd::PredNonzeroInt{}, ws, s);
    case GC_PRED_ODD: return dispatch_count(i, count, n, gcd::PredOdd{}, ws, s);
    default: return dispatch_count(i, count, n, gcd::PredEven{}, ws, s);
    }
}

cudaError_t launch_partition_cmp(const void *in, void *out, uint32_t *count_true, uint32_t n,
                                 gc_dtype dt, const CmpSpec &c, uint8_t *ws, cudaStream_t s,
                                 const LaunchOpts &o)
{
    auto *i = static_cast<const uint32_t *>(in);
    auto *u = static_cast<uint32_t *>(out);
    if (dt == GC_I32)
        return dispatch_partition(i, u, count_true, n,
                                  gcd::PredCmp<0>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o);
    if (dt == GC_U32)
        return dispatch_partition(i, u, count_true, n,
                                  gcd::PredCmp<1>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o);
    return dispatch_partition(i, u, count_true, n,
                              gcd::PredCmp<2>{c.lo, c.span, c.invert, c.is_mask, c.mask, c.value}, ws, s, o);
}

cudaError_t launch_split_radix(const uint32_t *keys_in, const uint32_t *vals_in,
                               uint32_t *keys_out, uint32_t *vals_out, uint32_t n, int begin_bit,
                               int end_bit, uint8_t *ws, cudaStream_t s, const LaunchOpts &o,
                               uint32_t key_neg, uint32_t key_flip)
{
    const bool keyed = (key_neg | key_flip) != 0u;
    const bool vals = vals_in != nullptr;
    const int passes = end_bit - begin_bit;
    cudaError_t e;
    if (passes == 0) {
        if (keys_out != keys_in) {
            e = cudaMemcpyAsync(keys_out, keys_in, size_t(n) * 4, cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return e;
        }
        if (vals && vals_out != vals_in)
            return cudaMemcpyAsync(vals_out, vals_in, size_t(n) * 4, cudaMemcpyDeviceToDevice, s);
        return cudaSuccess;
    }
    constexpr int RT = kReduceThreads;
    const int grid = reduce_grid(n, RT);
    if ((e = clear_accumulators(ws, s)) != cudaSuccess) return e;
    if (keyed) {
        if (aligned16(keys_in))
            bit_histogram_kernel<RT, true, true><<<grid, RT, 0, s>>>(keys_in, n, ws, key_neg, key_flip);
        else
            bit_histogram_kernel<RT, false, true><<<grid, RT, 0, s>>>(keys_in, n, ws, key_neg, key_flip);
    } else {
        if (aligned16(keys_in))
            bit_histogram_kernel<RT, true, false><<<grid, RT, 0, s>>>(keys_in, n, ws, 0u, 0u);
        else
            bit_histogram_kernel<RT, false, false><<<grid, RT, 0, s>>>(keys_in, n, ws, 0u, 0u);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(ws + radix_temp_offset(n));
    uint32_t *tmp_v = reinterpret_cast<uint32_t *>(ws + radix_temp_offset(n) + radix_temp_stride(n));
    const uint32_t *src_k = keys_in, *src_v = vals_in;
    const bool alias = keys_in == keys_out || (vals && vals_in == vals_out);
    if (alias && (passes & 1)) {
        // The first split would write over its own input: start from a copy.
        e = cudaMemcpyAsync(tmp_k, keys_in, size_t(n) * 4, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess && vals)
            e = cudaMemcpyAsync(tmp_v, vals_in, size_t(n) * 4, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return e;
        src_k = tmp_k;
        src_v = vals ? tmp_v : nullptr;
    }
    // Pass p publishes in region p % 2 of the status area (2 T words, which
    // the workspace holds) and clears the other region for pass p + 1, so
    // only the first pass clears its own words (behind its start barrier).
    // A pass that falls back to the one-tile-per-CTA kernels leaves both
    // regions to a memset.
    const uint32_t split_tiles = uint32_t(ceil_div(n, split_tile_elems()));
    const bool regions = 2ull * split_tiles <= max_tiles(n);
    bool fresh = true;  // the next pass's region still needs its own clear
    for (int p = 0; p < passes; ++p) {
        LaunchOpts po = o;
        if (regions) {
            po.reset_status = fresh;
            po.status_region = uint32_t(p % 2) * split_tiles;
            po.clear_region = uint32_t((p + 1) % 2) * split_tiles;
            po.clear_words = (p + 1 < passes) ? split_tiles : 0u;
        }
        bool piped = true;
        // The last pass writes the output; earlier ones alternate so that it does.
        const bool to_out = ((passes - 1 - p) % 2) == 0;
        uint32_t *dst_k = to_out ? keys_out : tmp_k;
        uint32_t *dst_v = vals ? (to_out ? vals_out : tmp_v) : nullptr;
        const int bit = begin_bit + p;
        const uint32_t *zeros = reinterpret_cast<const uint32_t *>(ws + kHdrBitZeros + 4 * bit);
        if (keyed) {
            const gcd::PredKeyBitClear pred{uint32_t(bit), key_neg, (key_flip >> bit) & 1u};
            e = vals ? run_partition_pass<gcd::PredKeyBitClear, true>(src_k, src_v, dst_k, dst_v, n, zeros, pred, ws, s, po, true, &piped)
                     : run_partition_pass<gcd::PredKeyBitClear, false>(src_k, nullptr, dst_k, nullptr, n, zeros, pred, ws, s, po, true, &piped);
        } else {
            const gcd::PredBitClear pred{uint32_t(bit)};
            e = vals ? run_partition_pass<gcd::PredBitClear, true>(src_k, src_v, dst_k, dst_v, n, zeros, pred, ws, s, po, true, &piped)
                     : run_partition_pass<gcd::PredBitClear, false>(src_k, nullptr, dst_k, nullptr, n, zeros, pred, ws, s, po, true, &piped);
        }
        if (e != cudaSuccess) return e;
        fresh = false;
        if (regions && !piped && p + 1 < passes &&
            (e = reset_tiles(ws, 2u * split_tiles, s, false)) != cudaSuccess)
            return e;
        src_k = dst_k;
        src_v = dst_v;
    }
    return cudaSuccess;
}

}  // namespace gch
