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
//      digit in shared memory as (key, payload) pairs, and writes each
//      digit's run to A[d * T + t] onwards, so consecutive threads store
//      consecutive addresses.  A full tile's keys and payloads are copied
//      into shared memory by the TMA unit while the counters are cleared,
//      so no payload load waits in the middle of the tile.
//
// Keys of int32 and float32 are sorted by the order-preserving key of
// PredKeyBitClear, x ^ (signfill(x) & neg) ^ flip: its digits are computed
// on the fly, by code specialised to the dtype's map, and the keys
// themselves move unchanged.
#include "gc_device.cuh"
#include "gc_internal.h"
#include "gc_pipe.cuh"

namespace {

using namespace gcd;

constexpr int kDigitBits = 8;
constexpr uint32_t kDigits = 1u << kDigitBits;
constexpr int kDigitThreads = 256;  // one thread per digit in the per-digit steps
constexpr int kDigitItems = 16;  // keys per thread
static_assert(kDigitThreads == int(kDigits), "one thread per digit");
static_assert(gch::kDigitTile == kDigitThreads * kDigitItems, "tile size");

// Digit of x under the order-preserving key map of its dtype: one of the
// key's bytes, taken with one permute (sel = 0x4440 | byte index).  uint32
// keys are their own key; int32 keys flip the sign bit; float32 keys flip
// every bit of a negative value and the sign bit of any other.
enum class KeyKind { U32, I32, F32 };

template <KeyKind K>
struct DigitOf {
    uint32_t sel;
    __device__ __forceinline__ uint32_t operator()(uint32_t x) const
    {
        uint32_t key = x;
        if constexpr (K == KeyKind::I32) key = x ^ 0x80000000u;
        if constexpr (K == KeyKind::F32) key = x ^ (uint32_t(int32_t(x) >> 31) | 0x80000000u);
        return __byte_perm(key, 0u, sel);
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
        m &= bal ^ (bit - 1u);
    }
    return m;
}

// Pass step 1: digit counts of tiles, written digit-major.  Each CTA counts
// kCountTiles consecutive tiles, with the keys of all of them loaded before
// the first is counted, by one shared-memory atomic per key.  The atomics'
// rate sets the kernel's pace, so their bank conflicts are kept low (below).
constexpr int kCountTiles = 2;  // 2 beat 1 and 4

template <class Dig, bool VEC>
__global__ void __launch_bounds__(kDigitThreads)
digit_count_kernel(const uint32_t *__restrict__ keys, uint32_t n, Dig dig,
                   uint32_t *__restrict__ counts, uint32_t tiles)
{
    // Eight sub-counts per digit, side by side, lane j counting into sub-count
    // j & 7: the lanes of one atomic instruction meet in a bank only when they
    // agree on j & 7 and on their digits' last two bits.
    __shared__ __align__(16) uint32_t s_hist[kCountTiles][kDigits][8];
    const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t)
#pragma unroll
        for (int j = 0; j < 8; ++j) (&s_hist[t][0][0])[j * kDigitThreads + tid] = 0u;

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
                if (full || i + q < n) atomicAdd(&s_hist[t][dig(x[t][r][q])][lane & 7], 1u);
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kCountTiles; ++t) {
        if (first + t < tiles) {
            const uint4 a = *reinterpret_cast<const uint4 *>(&s_hist[t][tid][0]);
            const uint4 b = *reinterpret_cast<const uint4 *>(&s_hist[t][tid][4]);
            const uint32_t c = (a.x + a.y) + (a.z + a.w) + ((b.x + b.y) + (b.z + b.w));
            counts[size_t(tid) * tiles + first + t] = c;
        }
    }
}

// The scatter's CTA: kScatThreads threads, kScatItems keys each; warp w owns
// keys [w * kScatSegment, (w + 1) * kScatSegment) of the tile, taken 32 at a
// time in order (key j of the warp's step s is lane j).  Threads below
// kDigits also do the per-digit steps.  256 threads x 16 keys at 4 CTAs per
// SM (64 registers, 42 KiB of shared memory each) beat 512 x 8 at 2
// or 3 CTAs per SM.
#ifndef GC_SCATTER_THREADS
#define GC_SCATTER_THREADS 256
#endif
constexpr int kScatThreads = GC_SCATTER_THREADS;
constexpr int kScatWarps = kScatThreads / 32;
constexpr int kScatItems = int(gch::kDigitTile) / kScatThreads;
constexpr uint32_t kScatSegment = 32u * kScatItems;
static_assert(kScatThreads >= int(kDigits) && kScatItems % 4 == 0, "scatter shape");

// Shared memory of the scatter (dynamic).  buf first receives the tile as
// staged (payloads in buf[0, T) and keys in buf[T, 2T), T = kDigitTile; keys
// only: buf[0, T)); once every thread holds its keys and payloads in
// registers it receives the tile sorted by digit, as (key, payload) pairs
// (keys only: keys).
template <bool VALS>
struct ScatterSmem {
    // Per warp and digit: the digit's count so far.  Entry kDigits is the
    // padding of the ragged tile.  After the scan: where the warp's first key
    // of the digit goes in the sorted tile.
    uint32_t cnt[kScatWarps][kDigits + 1];
    uint32_t adj[kDigits];  // output index of sorted position 0 of each digit's run
    uint32_t warp_sum[kDigits / 32];
    uint64_t bar[2];        // TMA completion: keys, payloads
    alignas(16) uint32_t buf[VALS ? 2 * gch::kDigitTile : gch::kDigitTile];
};

// Stable scatter of one tile by digit (FULL: all kDigitTile keys present;
// TMA: a full tile's keys and payloads are being copied into buf).
template <bool VALS, bool FULL, bool TMA, class Dig>
__device__ __forceinline__ void scatter_tile(const uint32_t *__restrict__ kin,
                                             const uint32_t *__restrict__ vin,
                                             uint32_t *__restrict__ kout, uint32_t *__restrict__ vout,
                                             uint32_t n, const Dig &dig, uint32_t tile,
                                             uint32_t valid, uint32_t glob, uint8_t *ws,
                                             uint64_t timeout_ns, ScatterSmem<VALS> &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = tile * gch::kDigitTile;
    auto staged = [&](int s) -> uint32_t {
        return uint32_t(warp) * kScatSegment + uint32_t(s) * 32u + uint32_t(lane);
    };

    // Without the TMA copies the tile is staged into buf here with plain loads.
    uint32_t *raw_k = sm.buf + (VALS ? gch::kDigitTile : 0u);
    if (!TMA) {
#pragma unroll
        for (int s = 0; s < kScatItems; ++s) {
            const uint32_t li = staged(s);
            raw_k[li] = (FULL || li < valid) ? kin[base + li] : 0u;
            if (VALS) sm.buf[li] = (FULL || li < valid) ? vin[base + li] : 0u;
        }
        __syncwarp();  // each warp reads back only its own segment
    } else {
        mbar_wait(&sm.bar[0], 0u, ws, timeout_ns);
    }
    // Digits: packed four to a word in a full tile; whole words, with the
    // padding value kDigits past the end, in the ragged one.
    uint32_t dg[FULL ? kScatItems / 4 : kScatItems];
#pragma unroll
    for (int s = 0; s < kScatItems; ++s) {
        const uint32_t li = staged(s);
        const uint32_t d = dig(raw_k[li]);
        if (FULL) {
            if ((s & 3) == 0) dg[s >> 2] = d;
            else dg[s >> 2] |= d << (8 * (s & 3));
        } else {
            dg[s] = li < valid ? d : kDigits;
        }
    }
    auto digit = [&](int s) -> uint32_t {
        return FULL ? __byte_perm(dg[s >> 2], 0u, 0x4440u | uint32_t(s & 3)) : dg[s];
    };

    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t *wcnt = sm.cnt[warp];
    uint32_t rank2[kScatItems / 2];
    // Stable rank within the warp's segment: the peers of a key are the
    // lanes of its step with the same digit; the step's leader for each digit
    // (its lowest lane) adds the group to the warp's counter and keeps the old
    // value for its peers.  Ranks (below kScatSegment) are kept two to a word.
#pragma unroll
    for (int s = 0; s < kScatItems; ++s) {
        const uint32_t ds = digit(s);
        const uint32_t peers = digit_peers<FULL ? kDigitBits : kDigitBits + 1>(ds);
        uint32_t before = 0u;
        if ((peers & lt_mask) == 0u) {
            before = wcnt[ds];
            wcnt[ds] = before + uint32_t(__popc(peers));
        }
        // The next step's leader for this digit may be another lane: order
        // this step's counter writes before its reads.
        __syncwarp();
        const uint32_t r = __shfl_sync(kFullMask, before, __ffs(peers) - 1) + uint32_t(__popc(peers & lt_mask));
        if ((s & 1) == 0) rank2[s >> 1] = r;
        else rank2[s >> 1] |= r << 16;
    }
    __syncthreads();

    // Per digit (threads below kDigits, thread = digit): exclusive scan over
    // the warps, then over the digits for the tile-local run starts.
    uint32_t total = 0u, incl = 0u;
    if (tid < int(kDigits)) {
#pragma unroll
        for (int w = 0; w < kScatWarps; ++w) {
            const uint32_t c = sm.cnt[w][tid];
            sm.cnt[w][tid] = total;
            total += c;
        }
        incl = total;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) sm.warp_sum[warp] = incl;
    }
    // The keys and payloads, read back in the order of the ranks before the
    // sorted tile overwrites them.
    if (TMA && VALS) mbar_wait(&sm.bar[1], 0u, ws, timeout_ns);
    uint32_t k[kScatItems], v[VALS ? kScatItems : 1];
#pragma unroll
    for (int s = 0; s < kScatItems; ++s) {
        const uint32_t li = staged(s);
        k[s] = raw_k[li];
        if (VALS) v[VALS ? s : 0] = sm.buf[li];
    }
    __syncthreads();
    if (tid < int(kDigits)) {
        uint32_t wbase = 0u;
#pragma unroll
        for (int w = 0; w < int(kDigits / 32); ++w) wbase += (w < warp) ? sm.warp_sum[w] : 0u;
        const uint32_t start = wbase + incl - total;
#pragma unroll
        for (int w = 0; w < kScatWarps; ++w) sm.cnt[w][tid] += start;
        sm.adj[tid] = glob - start;
    }
    __syncthreads();

    // Tile-local sort by digit in shared memory.  With payloads each key's
    // digit is computed again here, so the packed digits die after the
    // ranking and the payloads fit in registers without spills (5.49 -> 5.34
    // ms per float32 sort with payloads at 2^28); keys alone keep them.
#pragma unroll
    for (int s = 0; s < kScatItems; ++s) {
        const uint32_t ds = VALS ? (FULL || staged(s) < valid ? dig(k[s]) : kDigits) : digit(s);
        if (FULL || ds < kDigits) {
            const uint32_t pos = wcnt[ds] + ((rank2[s >> 1] >> (16 * (s & 1))) & 0xffffu);
            if (VALS) reinterpret_cast<uint2 *>(sm.buf)[pos] = make_uint2(k[s], v[VALS ? s : 0]);
            else sm.buf[pos] = k[s];
        }
    }
    __syncthreads();

    // Write out in sorted order: position i of the tile belongs to the run of
    // its digit, which starts at output index adj[digit] + (its start here).
#pragma unroll
    for (int s = 0; s < kScatItems; ++s) {
        const uint32_t i = uint32_t(s) * kScatThreads + uint32_t(tid);
        if (FULL || i < valid) {
            uint32_t key, val = 0u;
            if (VALS) {
                const uint2 kv = reinterpret_cast<const uint2 *>(sm.buf)[i];
                key = kv.x;
                val = kv.y;
            } else {
                key = sm.buf[i];
            }
            const uint32_t g = sm.adj[dig(key)] + i;
            if (g < n) {
                __stcs(kout + g, key);
                if (VALS) __stcs(vout + g, val);
            } else {
                record_error(ws, kDeviceCheckCode, tile);  // a corrupted count table
            }
        }
    }
}

// Pass step 3: stable scatter of one tile by digit.  offsets[d * T + t] is
// where tile t's run of digit d starts in the output.
#ifndef GC_DIGIT_SCATTER_MIN_BLOCKS
#define GC_DIGIT_SCATTER_MIN_BLOCKS 4
#endif

template <class Dig, bool VALS, bool TMA>
__global__ void __launch_bounds__(kScatThreads, GC_DIGIT_SCATTER_MIN_BLOCKS)
digit_scatter_kernel(const uint32_t *__restrict__ kin, const uint32_t *__restrict__ vin,
                     uint32_t *__restrict__ kout, uint32_t *__restrict__ vout, uint32_t n,
                     Dig dig, const uint32_t *__restrict__ offsets, uint32_t tiles,
                     uint8_t *ws, uint64_t timeout_ns)
{
    extern __shared__ __align__(16) uint8_t scatter_smem[];
    ScatterSmem<VALS> &sm = *reinterpret_cast<ScatterSmem<VALS> *>(scatter_smem);
    const int tid = threadIdx.x;
    const uint32_t tile = blockIdx.x;
    const uint32_t valid = min(gch::kDigitTile, n - tile * gch::kDigitTile);
    const bool full = valid == gch::kDigitTile;
    if (TMA && full && tid == 0) {
        // Payloads into buf[0, T), keys into buf[T, 2T) (T = kDigitTile).
        constexpr uint32_t kBytes = gch::kDigitTile * 4u;
        const uint32_t base = tile * gch::kDigitTile;
        mbar_init(&sm.bar[0], 1u);
        if (VALS) mbar_init(&sm.bar[1], 1u);
        fence_barrier_init();
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sm.bar[0], kBytes);
        bulk_load(sm.buf + (VALS ? gch::kDigitTile : 0u), kin + base, kBytes, &sm.bar[0]);
        if (VALS) {
            mbar_arrive_expect_tx(&sm.bar[1], kBytes);
            bulk_load(sm.buf, vin + base, kBytes, &sm.bar[1]);
        }
    }
    for (uint32_t i = uint32_t(tid); i < uint32_t(kScatWarps) * (kDigits + 1u); i += kScatThreads)
        (&sm.cnt[0][0])[i] = 0u;
    const uint32_t glob = tid < int(kDigits) ? offsets[size_t(tid) * tiles + tile] : 0u;
    __syncthreads();  // counters cleared, barriers initialised
    if (!full)
        scatter_tile<VALS, false, false>(kin, vin, kout, vout, n, dig, tile, valid, glob, ws, timeout_ns, sm);
    else if (TMA)
        scatter_tile<VALS, true, true>(kin, vin, kout, vout, n, dig, tile, valid, glob, ws, timeout_ns, sm);
    else
        scatter_tile<VALS, true, false>(kin, vin, kout, vout, n, dig, tile, valid, glob, ws, timeout_ns, sm);
}

template <class Dig, bool VALS, bool TMA>
cudaError_t launch_scatter(const uint32_t *kin, const uint32_t *vin, uint32_t *kout, uint32_t *vout,
                           uint32_t n, const Dig &dig, const uint32_t *table, uint32_t tiles,
                           uint8_t *ws, cudaStream_t s, const gch::LaunchOpts &o)
{
    constexpr size_t kSmem = sizeof(ScatterSmem<VALS>);
    auto kern = digit_scatter_kernel<Dig, VALS, TMA>;
    // Sets the kernel's shared-memory limit, once per device.
    if (gch::persistent_grid(reinterpret_cast<const void *>(kern), kScatThreads, kSmem, tiles) <= 0)
        return cudaErrorInvalidConfiguration;
    kern<<<tiles, kScatThreads, kSmem, s>>>(kin, vin, kout, vout, n, dig, table, tiles, ws, o.timeout_ns);
    return cudaGetLastError();
}

// The four passes of one sort, keys mapped to their order-preserving keys
// by Dig.
template <KeyKind K>
cudaError_t sort_digits(const uint32_t *keys_in, const uint32_t *vals_in, uint32_t *keys_out,
                        uint32_t *vals_out, uint32_t n, uint8_t *ws, cudaStream_t s,
                        const gch::LaunchOpts &o)
{
    using Dig = DigitOf<K>;
    const bool vals = vals_in != nullptr;
    const uint32_t tiles = uint32_t(gch::ceil_div(n, gch::kDigitTile));
    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(ws + gch::radix_temp_offset(n));
    uint32_t *tmp_v = reinterpret_cast<uint32_t *>(ws + gch::radix_temp_offset(n) + gch::radix_temp_stride(n));
    uint32_t *table = reinterpret_cast<uint32_t *>(ws + gch::digit_table_offset(n));
    uint32_t *scan_total = reinterpret_cast<uint32_t *>(ws + gch::kHdrDigitScanTotal);
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
        const Dig dig{0x4440u | uint32_t(p)};  // byte p of the key
        const uint32_t count_grid = uint32_t(gch::ceil_div(tiles, kCountTiles));
        if (gch::aligned16(src_k))
            digit_count_kernel<Dig, true><<<count_grid, kDigitThreads, 0, s>>>(src_k, n, dig, table, tiles);
        else
            digit_count_kernel<Dig, false><<<count_grid, kDigitThreads, 0, s>>>(src_k, n, dig, table, tiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        e = gch::launch_scan(table, table, scan_total, tiles * kDigits, GC_U32, ws, s, o, false);
        if (e != cudaSuccess) return e;
        // Full tiles are staged by TMA when the sources are 16-byte aligned.
        const bool tma = gch::aligned16(src_k) && (!vals || gch::aligned16(src_v));
        if (vals)
            e = tma ? launch_scatter<Dig, true, true>(src_k, src_v, dst_k, dst_v, n, dig, table, tiles, ws, s, o)
                    : launch_scatter<Dig, true, false>(src_k, src_v, dst_k, dst_v, n, dig, table, tiles, ws, s, o);
        else
            e = tma ? launch_scatter<Dig, false, true>(src_k, nullptr, dst_k, nullptr, n, dig, table, tiles, ws, s, o)
                    : launch_scatter<Dig, false, false>(src_k, nullptr, dst_k, nullptr, n, dig, table, tiles, ws, s, o);
        if (e != cudaSuccess) return e;
        src_k = dst_k;
        src_v = dst_v;
    }
    return cudaSuccess;
}

}  // namespace

namespace gch {

cudaError_t launch_radix_sort_digits(const uint32_t *keys_in, const uint32_t *vals_in,
                                     uint32_t *keys_out, uint32_t *vals_out, uint32_t n,
                                     uint32_t key_neg, uint32_t key_flip, uint8_t *ws,
                                     cudaStream_t s, const LaunchOpts &o)
{
    // The three order-preserving key maps x ^ (signfill(x) & neg) ^ flip.
    if (key_neg == 0u && key_flip == 0u)
        return sort_digits<KeyKind::U32>(keys_in, vals_in, keys_out, vals_out, n, ws, s, o);
    if (key_neg == 0u && key_flip == 0x80000000u)
        return sort_digits<KeyKind::I32>(keys_in, vals_in, keys_out, vals_out, n, ws, s, o);
    if (key_neg == 0x7FFFFFFFu && key_flip == 0x80000000u)
        return sort_digits<KeyKind::F32>(keys_in, vals_in, keys_out, vals_out, n, ws, s, o);
    return cudaErrorInvalidValue;
}

}  // namespace gch
