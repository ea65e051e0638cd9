// radix.cu -- LSD radix sort by 8-bit digits: the multi-way generalisation of
// the one-bit split.
//
// "CIS 565 Project 2: Stream Compaction" builds its radix sort from one
// stable two-way split per bit, each addressed by a scan of the predicate.
// With a digit of 8 bits a pass splits the keys stably into 256 buckets
// instead of 2, and the scan that addresses them runs over the per-tile
// digit counts instead of the per-element flags; four passes sort 32-bit
// keys.  Each pass is three launches:
//
//   1. digit_count_kernel: every tile of kDigitTile keys counts its digits
//      and writes them digit-major, A[d * T + t] (T tiles).
//   2. the exclusive scan of A (this library's own scan kernel): A[d * T + t]
//      becomes the number of keys that go before tile t's first key of digit
//      d, namely every key of a smaller digit plus the keys of digit d in
//      earlier tiles.  One scan yields both the bucket bases and the
//      per-tile offsets.
//   3. digit_scatter_kernel: every tile ranks its keys stably within the
//      tile (warp by warp, 32 keys at a time: peers found by one ballot per
//      digit bit, per-warp digit counters in shared memory), sorts them by
//      digit in shared memory, and writes each digit's run to A[d * T + t]
//      onwards, so consecutive threads store consecutive addresses.
//
// Keys of int32 and float32 are sorted by the order-preserving key of
// PredKeyBitClear, x ^ (signfill(x) & neg) ^ flip: its digits are computed
// on the fly and the keys themselves move unchanged.
#include "gc_device.cuh"
#include "gc_internal.h"

namespace {

using namespace gcd;

constexpr int kDigitBits = 8;
constexpr uint32_t kDigits = 1u << kDigitBits;
constexpr int kDigitThreads = 256;  // one thread per digit in the per-digit steps
constexpr int kDigitWarps = kDigitThreads / 32;
constexpr int kDigitItems = 16;  // keys per thread
constexpr uint32_t kSegment = 32u * kDigitItems;  // keys per warp, in order
static_assert(kDigitThreads == int(kDigits), "one thread per digit");
static_assert(gch::kDigitTile == kDigitThreads * kDigitItems, "tile size");

// Digit of x at `shift` under the order-preserving key map.
struct DigitOf {
    uint32_t neg, flip, shift;
    __device__ __forceinline__ uint32_t operator()(uint32_t x) const
    {
        const uint32_t key = x ^ ((uint32_t(int32_t(x) >> 31) & neg) ^ flip);
        return (key >> shift) & (kDigits - 1u);
    }
};

// Lanes of the warp whose digit equals this lane's: one ballot per bit of d
// (BITS bits; the ragged last tile adds one for its padding value kDigits),
// each narrowing the set to the lanes that agree on that bit.
template <int BITS>
__device__ __forceinline__ uint32_t digit_peers(uint32_t d)
{
    uint32_t m = kFullMask;
#pragma unroll
    for (int b = 0; b < BITS; ++b) {
        const uint32_t bit = (d >> b) & 1u;
        const uint32_t bal = __ballot_sync(kFullMask, bit != 0u);
        m &= bal ^ (bit - 1u);  // bal where my bit is 1, ~bal where it is 0
    }
    return m;
}

// Pass step 1: digit counts of tiles, written digit-major.  Each CTA counts
// kCountTiles consecutive tiles, with the keys of all of them loaded before
// the first is counted; shared-memory histograms are private to a warp and
// a lane parity, so two lanes of one atomic instruction collide only when
// they share both parity and digit.
constexpr int kCountTiles = 2;
constexpr int kCountHists = 2 * kDigitWarps;

template <bool VEC>
__global__ void __launch_bounds__(kDigitThreads)
digit_count_kernel(const uint32_t *__restrict__ keys, uint32_t n, DigitOf dig,
                   uint32_t *__restrict__ counts, uint32_t tiles)
{
    __shared__ uint32_t s_hist[kCountTiles][kCountHists][kDigits];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = 2 * warp + (lane & 1);
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t)
#pragma unroll
        for (int w = 0; w < kCountHists; ++w) s_hist[t][w][tid] = 0u;

    constexpr int kVecs = kDigitItems / 4;  // 4-key vectors per thread per tile
    uint32_t x[kCountTiles][kVecs][4];
    const uint32_t first = blockIdx.x * kCountTiles;
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t)
#pragma unroll
        for (int r = 0; r < kVecs; ++r) {
            const uint32_t i = (first + t) * gch::kDigitTile + uint32_t(r) * (4u * kDigitThreads) +
                               4u * uint32_t(tid);
            load4<VEC>(keys, i, n, 0u, x[t][r]);
        }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t) {
        const uint32_t base = (first + t) * gch::kDigitTile;
        const bool full = base + gch::kDigitTile <= n;
#pragma unroll
        for (int r = 0; r < kVecs; ++r) {
            const uint32_t i = base + uint32_t(r) * (4u * kDigitThreads) + 4u * uint32_t(tid);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (full || i + q < n) atomicAdd(&s_hist[t][h][dig(x[t][r][q])], 1u);
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t) {
        if (first + t < tiles) {
            uint32_t c = 0u;
#pragma unroll
            for (int w = 0; w < kCountHists; ++w) c += s_hist[t][w][tid];
            counts[size_t(tid) * tiles + first + t] = c;
        }
    }
}

struct ScatterSmem {
    uint32_t cnt[kDigitWarps][kDigits];  // per-warp running counts, then offsets
    uint32_t start[kDigits];             // tile-local start of each digit's run
    uint32_t glob[kDigits];              // global start of each digit's run
    uint32_t warp_sum[kDigitWarps];
    uint32_t keys[gch::kDigitTile];
};

// Stable scatter of one tile by digit (FULL: all kDigitTile keys present).
template <bool VALS, bool FULL>
__device__ __forceinline__ void scatter_tile(const uint32_t *__restrict__ kin,
                                             const uint32_t *__restrict__ vin,
                                             uint32_t *__restrict__ kout, uint32_t *__restrict__ vout,
                                             uint32_t n, const DigitOf &dig, uint32_t tile,
                                             uint32_t valid, uint8_t *ws, ScatterSmem &sm,
                                             uint32_t *s_vals)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = tile * gch::kDigitTile;

    // Warp w owns keys [w * kSegment, (w + 1) * kSegment) of the tile, taken
    // 32 at a time in order: key j of the warp's step s is lane j.
    uint32_t k[kDigitItems];
#pragma unroll
    for (int s = 0; s < kDigitItems; ++s) {
        const uint32_t li = uint32_t(warp) * kSegment + uint32_t(s) * 32u + uint32_t(lane);
        k[s] = (FULL || li < valid) ? kin[base + li] : 0u;
    }
    // Digits: packed four to a word in a full tile; whole words, with the
    // padding value kDigits past the end, in the ragged one.
    uint32_t dg[FULL ? kDigitItems / 4 : kDigitItems];
#pragma unroll
    for (int s = 0; s < kDigitItems; ++s) {
        if (FULL) {
            if ((s & 3) == 0) dg[s >> 2] = 0u;
            dg[s >> 2] |= dig(k[s]) << (8 * (s & 3));
        } else {
            const uint32_t li = uint32_t(warp) * kSegment + uint32_t(s) * 32u + uint32_t(lane);
            dg[s] = li < valid ? dig(k[s]) : kDigits;
        }
    }
    auto digit = [&](int s) -> uint32_t {
        return FULL ? (dg[s >> 2] >> (8 * (s & 3))) & (kDigits - 1u) : dg[s];
    };
    __syncthreads();  // the counters are cleared

    // Stable rank within the warp's segment: the peers of a key are the
    // lanes of its step with the same digit; the step's leader for each digit
    // (its lowest lane) adds the group to the warp's counter and keeps the old
    // value for its peers.  Ranks (below kSegment) are kept two to a word.
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t rank2[kDigitItems / 2];
#pragma unroll
    for (int s = 0; s < kDigitItems; ++s) {
        const uint32_t ds = digit(s);
        const uint32_t peers = digit_peers<FULL ? kDigitBits : kDigitBits + 1>(ds);
        uint32_t before = 0u;
        if ((peers & lt_mask) == 0u && (FULL || ds < kDigits)) {
            before = sm.cnt[warp][ds];
            sm.cnt[warp][ds] = before + uint32_t(__popc(peers));
        }
        // The next step's leader for this digit may be another lane: order
        // this step's counter writes before its reads.
        __syncwarp();
        const uint32_t r = __shfl_sync(kFullMask, before, __ffs(peers) - 1) + uint32_t(__popc(peers & lt_mask));
        if ((s & 1) == 0) rank2[s >> 1] = r;
        else rank2[s >> 1] |= r << 16;
    }
    __syncthreads();
    // The payloads are read only now, when the ranking no longer needs the
    // registers; their latency overlaps the scans below.
    uint32_t v[VALS ? kDigitItems : 1];
    if (VALS) {
#pragma unroll
        for (int s = 0; s < kDigitItems; ++s) {
            const uint32_t li = uint32_t(warp) * kSegment + uint32_t(s) * 32u + uint32_t(lane);
            v[VALS ? s : 0] = (FULL || li < valid) ? vin[base + li] : 0u;
        }
    }

    // Per digit (thread tid = digit): exclusive scan over the warps, then over
    // the digits for the tile-local run starts.
    uint32_t total = 0u;
#pragma unroll
    for (int w = 0; w < kDigitWarps; ++w) {
        const uint32_t c = sm.cnt[w][tid];
        sm.cnt[w][tid] = total;
        total += c;
    }
    uint32_t incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t wbase = 0u;
#pragma unroll
    for (int w = 0; w < kDigitWarps; ++w) wbase += (w < warp) ? sm.warp_sum[w] : 0u;
    sm.start[tid] = wbase + incl - total;
    __syncthreads();

    // Tile-local sort by digit in shared memory.
#pragma unroll
    for (int s = 0; s < kDigitItems; ++s) {
        const uint32_t ds = digit(s);
        if (FULL || ds < kDigits) {
            const uint32_t pos = sm.start[ds] + sm.cnt[warp][ds] + ((rank2[s >> 1] >> (16 * (s & 1))) & 0xffffu);
            sm.keys[pos] = k[s];
            if (VALS) s_vals[pos] = v[VALS ? s : 0];
        }
    }
    __syncthreads();

    // Write out in sorted order: position i of the tile belongs to the run of
    // its digit, which starts at start[digit] here and glob[digit] there.
#pragma unroll
    for (int s = 0; s < kDigitItems; ++s) {
        const uint32_t i = uint32_t(s) * kDigitThreads + uint32_t(tid);
        if (FULL || i < valid) {
            const uint32_t key = sm.keys[i];
            const uint32_t dd = dig(key);
            const uint32_t g = sm.glob[dd] + (i - sm.start[dd]);
            if (g < n) {
                __stcs(kout + g, key);
                if (VALS) __stcs(vout + g, s_vals[i]);
            } else {
                record_error(ws, kDeviceCheckCode, tile);  // a corrupted count table
            }
        }
    }
}

// Pass step 3: stable scatter of one tile by digit.  offsets[d * T + t] is
// where tile t's run of digit d starts in the output.
// Resident CTAs per SM the scatter is compiled for (registers: 4 -> 64): the
// kernel is latency-bound, and 4 CTAs per SM beat 2, 3 and 5.
#ifndef GC_DIGIT_SCATTER_MIN_BLOCKS
#define GC_DIGIT_SCATTER_MIN_BLOCKS 4
#endif

template <bool VALS>
__global__ void __launch_bounds__(kDigitThreads, GC_DIGIT_SCATTER_MIN_BLOCKS)
digit_scatter_kernel(const uint32_t *__restrict__ kin, const uint32_t *__restrict__ vin,
                     uint32_t *__restrict__ kout, uint32_t *__restrict__ vout, uint32_t n,
                     DigitOf dig, const uint32_t *__restrict__ offsets, uint32_t tiles,
                     uint8_t *ws)
{
    __shared__ ScatterSmem sm;
    __shared__ uint32_t s_vals[VALS ? gch::kDigitTile : 1];
    const int tid = threadIdx.x;
    const uint32_t tile = blockIdx.x;
    const uint32_t valid = min(gch::kDigitTile, n - tile * gch::kDigitTile);
#pragma unroll
    for (int w = 0; w < kDigitWarps; ++w) sm.cnt[w][tid] = 0u;
    sm.glob[tid] = offsets[size_t(tid) * tiles + tile];
    if (valid == gch::kDigitTile)
        scatter_tile<VALS, true>(kin, vin, kout, vout, n, dig, tile, valid, ws, sm, s_vals);
    else
        scatter_tile<VALS, false>(kin, vin, kout, vout, n, dig, tile, valid, ws, sm, s_vals);
}

}  // namespace

namespace gch {

cudaError_t launch_radix_sort_digits(const uint32_t *keys_in, const uint32_t *vals_in,
                                     uint32_t *keys_out, uint32_t *vals_out, uint32_t n,
                                     uint32_t key_neg, uint32_t key_flip, uint8_t *ws,
                                     cudaStream_t s, const LaunchOpts &o)
{
    const bool vals = vals_in != nullptr;
    const uint32_t tiles = uint32_t(ceil_div(n, kDigitTile));
    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(ws + radix_temp_offset(n));
    uint32_t *tmp_v = reinterpret_cast<uint32_t *>(ws + radix_temp_offset(n) + radix_temp_stride(n));
    uint32_t *table = reinterpret_cast<uint32_t *>(ws + digit_table_offset(n));
    uint32_t *scan_total = reinterpret_cast<uint32_t *>(ws + kHdrDigitScanTotal);
    constexpr int kPasses = 32 / kDigitBits;
    static_assert(kPasses % 2 == 0, "an even pass count ends in the output buffers");

    const uint32_t *src_k = keys_in, *src_v = vals_in;
    cudaError_t e = cudaSuccess;
    for (int p = 0; p < kPasses; ++p) {
        // Even passes write the workspace, odd ones the output, so the last
        // pass lands in the output and no pass overwrites its own input
        // (also when the input is the output).
        uint32_t *dst_k = (p % 2 == 0) ? tmp_k : keys_out;
        uint32_t *dst_v = vals ? ((p % 2 == 0) ? tmp_v : vals_out) : nullptr;
        const DigitOf dig{key_neg, key_flip, uint32_t(p * kDigitBits)};
        const uint32_t count_grid = uint32_t(ceil_div(tiles, kCountTiles));
        if (aligned16(src_k))
            digit_count_kernel<true><<<count_grid, kDigitThreads, 0, s>>>(src_k, n, dig, table, tiles);
        else
            digit_count_kernel<false><<<count_grid, kDigitThreads, 0, s>>>(src_k, n, dig, table, tiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        e = launch_scan(table, table, scan_total, tiles * kDigits, GC_U32, ws, s, o, false);
        if (e != cudaSuccess) return e;
        if (vals)
            digit_scatter_kernel<true><<<tiles, kDigitThreads, 0, s>>>(src_k, src_v, dst_k, dst_v, n,
                                                                       dig, table, tiles, ws);
        else
            digit_scatter_kernel<false><<<tiles, kDigitThreads, 0, s>>>(src_k, nullptr, dst_k, nullptr,
                                                                        n, dig, table, tiles, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        src_k = dst_k;
        src_v = dst_v;
    }
    return cudaSuccess;
}

}  // namespace gch
