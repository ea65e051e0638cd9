// gc_device.cuh -- device building blocks shared by every libgc kernel:
// the workspace layout, per-tile status words, the decoupled look-back, the
// tile loads and the predicates.
//
// The single-pass structure follows "The CUDA Handbook, ch. 13: Stream
// compaction" (Listing 13-17): a CTA takes the next tile id from a global
// counter, so every lower-numbered tile has already been taken by a CTA that
// is running or finished; it reduces its tile, publishes the tile aggregate,
// looks back over its predecessors' status for its exclusive prefix, and
// publishes its inclusive prefix.  The look-back itself is the one of
// Merrill and Garland, "Single-pass Parallel Prefix Scan with Decoupled
// Look-back" (NVIDIA technical report NVR-2016-002), which that chapter
// refers to and does not reprint; the code below is written from that
// description for one warp of 32 lanes reading 32 predecessors at a time.
#pragma once

#include <cstdint>

namespace gcd {

// ---------------------------------------------------------------- workspace
//
// [0, 512)             header (offsets below)
// [512, 512 + 8 T)     one 64-bit status word per tile, T = tiles of the call
// then, float32 scan:  one double inclusive prefix per tile
// radix:               the key and payload ping-pong buffers (see radix.cu)
//
// Each call clears the tile counter and its T status words with one
// cudaMemsetAsync of [kTileCtrOff, 512 + 8 T) before its kernel, so a status
// word is never read with contents from an earlier call.
constexpr uint32_t kHdrError = 0;        // u32: first device failure (gc_status), 0 = none
constexpr uint32_t kHdrErrorTile = 4;    // u32: tile whose wait gave up
constexpr uint32_t kHdrReduceCtr = 8;    // u32: CTAs finished in a count pre-pass (self-resetting)
constexpr uint32_t kHdrCountTrue = 12;   // u32: partition: elements the predicate keeps
constexpr uint32_t kHdrCountAcc = 16;    // u32: count pre-pass accumulator (reset by the last CTA)
constexpr uint32_t kHdrBitAcc = 64;      // u32[32]: radix: keys with bit b set, accumulating
constexpr uint32_t kHdrBitZeros = 192;   // u32[32]: radix: keys with bit b clear
constexpr uint32_t kTileCtrOff = 504;    // u32: next tile id (cleared with the status words)
constexpr uint32_t kStatusOff = 512;
constexpr uint32_t kHeaderBytes = 512;

__device__ __forceinline__ uint32_t *hdr_u32(uint8_t *ws, uint32_t off)
{
    return reinterpret_cast<uint32_t *>(ws + off);
}

// ---------------------------------------------------------------- status words
//
// One 64-bit word per tile: low half the value (a uint32 count or sum, or
// float32 bits), high half the flag.  One aligned 64-bit store publishes
// value and flag together, so a reader never sees one without the other.
// 16 words share a 128-byte line, so one warp reads 32 predecessors with two
// line requests.
constexpr uint32_t kFlagNone = 0;       // not yet published (the cleared state)
constexpr uint32_t kFlagAggregate = 1;  // value = this tile's own total
constexpr uint32_t kFlagPrefix = 2;     // value = total of tiles 0..this one

__device__ __forceinline__ uint64_t pack_status(uint32_t value, uint32_t flag)
{
    return (uint64_t(flag) << 32) | value;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint64_t *p, uint64_t v)
{
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ double ld_relaxed_gpu_f64(const double *p)
{
    double v;
    asm volatile("ld.relaxed.gpu.global.f64 %0, [%1];" : "=d"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_f64(double *p, double v)
{
    asm volatile("st.relaxed.gpu.global.f64 [%0], %1;" ::"l"(p), "d"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Records the first device-side failure in the workspace header.
__device__ __forceinline__ void record_error(uint8_t *ws, uint32_t code, uint32_t tile)
{
    if (atomicCAS(hdr_u32(ws, kHdrError), 0u, code) == 0u) {
        atomicExch(hdr_u32(ws, kHdrErrorTile), tile);
    }
}

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr uint32_t kTimeoutCode = 6;      // GC_ERR_TIMEOUT
constexpr uint32_t kDeviceCheckCode = 7;  // GC_ERR_DEVICE_CHECK

template <class V>
__device__ __forceinline__ V warp_sum(V v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

// Lane mask of lanes whose status matters in one look-back window: every
// lane up to and including the nearest (lowest-lane) prefix, or all 32 if no
// lane holds a prefix.
__device__ __forceinline__ uint32_t lanes_up_to_first(uint32_t prefix_mask)
{
    if (prefix_mask == 0u) return kFullMask;
    const uint32_t lowest = prefix_mask & (0u - prefix_mask);
    return lowest == 0x80000000u ? kFullMask : (lowest << 1) - 1u;
}

// Waits for one 32-tile window to resolve.  Lane l reads the status of tile
// win - l (a virtual prefix of 0 below tile 0).  Returns when every lane up
// to the nearest prefix has published something; on timeout records the
// error and returns with the unpublished lanes read as 0.
// Out: value/flag of this lane, the prefix-lane mask.
__device__ __forceinline__ void wait_window(const uint64_t *status, int64_t win,
                                            uint32_t &value, uint32_t &flag,
                                            uint32_t &prefix_mask, uint8_t *ws,
                                            uint32_t tile, uint64_t timeout_ns,
                                            uint64_t &t_start, bool &timed_out)
{
    const int lane = threadIdx.x & 31;
    const int64_t j = win - lane;
    uint32_t spins = 0;
    for (;;) {
        if (j >= 0) {
            const uint64_t w = ld_relaxed_gpu(status + j);
            value = uint32_t(w);
            flag = uint32_t(w >> 32);
        } else {
            value = 0u;
            flag = kFlagPrefix;
        }
        prefix_mask = __ballot_sync(kFullMask, flag == kFlagPrefix);
        const uint32_t missing = __ballot_sync(kFullMask, flag == kFlagNone);
        if ((missing & lanes_up_to_first(prefix_mask)) == 0u) return;
        // Some predecessor in range has not published yet: back off and retry.
        if (spins == 0) t_start = global_timer_ns();
        ++spins;
        // Lane 0's clock decides, so the whole warp leaves together.
        if ((spins & 15u) == 0u &&
            __shfl_sync(kFullMask, int(global_timer_ns() - t_start > timeout_ns), 0)) {
            if (lane == 0) record_error(ws, kTimeoutCode, tile);
            if (flag == kFlagNone) value = 0u;
            timed_out = true;
            return;
        }
        __nanosleep(spins < 8 ? 20 : 100);
    }
}

// Decoupled look-back for uint32 sums (counts and integer scans), run by one
// full warp.  Publishes `aggregate` for `tile`, finds the exclusive prefix,
// publishes the inclusive prefix, and returns the exclusive prefix to every
// lane.
__device__ __forceinline__ uint32_t lookback_u32(uint64_t *status, uint32_t tile,
                                                 uint32_t aggregate, uint8_t *ws,
                                                 uint64_t timeout_ns)
{
    const int lane = threadIdx.x & 31;
    if (tile == 0) {
        if (lane == 0) st_relaxed_gpu(status, pack_status(aggregate, kFlagPrefix));
        return 0u;
    }
    if (lane == 0) st_relaxed_gpu(status + tile, pack_status(aggregate, kFlagAggregate));
    uint32_t exclusive = 0u;
    int64_t win = int64_t(tile) - 1;
    uint64_t t_start = 0;
    bool timed_out = false;
    for (;;) {
        uint32_t value, flag, prefix_mask;
        wait_window(status, win, value, flag, prefix_mask, ws, tile, timeout_ns, t_start,
                    timed_out);
        const uint32_t use = lanes_up_to_first(prefix_mask);
        exclusive += warp_sum(((use >> lane) & 1u) ? value : 0u);
        if (prefix_mask != 0u || timed_out) break;
        win -= 32;
    }
    if (lane == 0) st_relaxed_gpu(status + tile, pack_status(exclusive + aggregate, kFlagPrefix));
    return exclusive;
}

// Decoupled look-back for float32 sums.  Tile aggregates travel as float32
// in the status word; the running prefix travels as a double in a side array
// (prefix64), written before the prefix flag is released, so the carry from
// tile to tile accumulates in double and its rounding does not grow with the
// number of tiles.  Returns the exclusive prefix as a double to every lane.
__device__ __forceinline__ double lookback_f32(uint64_t *status, double *prefix64,
                                               uint32_t tile, float aggregate,
                                               uint8_t *ws, uint64_t timeout_ns)
{
    const int lane = threadIdx.x & 31;
    if (tile == 0) {
        if (lane == 0) {
            st_relaxed_gpu_f64(prefix64, double(aggregate));
            st_release_gpu(status, pack_status(__float_as_uint(aggregate), kFlagPrefix));
        }
        return 0.0;
    }
    if (lane == 0)
        st_relaxed_gpu(status + tile, pack_status(__float_as_uint(aggregate), kFlagAggregate));
    double exclusive = 0.0;
    int64_t win = int64_t(tile) - 1;
    uint64_t t_start = 0;
    bool timed_out = false;
    for (;;) {
        uint32_t value, flag, prefix_mask;
        wait_window(status, win, value, flag, prefix_mask, ws, tile, timeout_ns, t_start,
                    timed_out);
        const uint32_t use = lanes_up_to_first(prefix_mask);
        double mine = 0.0;
        if ((use >> lane) & 1u) {
            const int64_t j = win - lane;
            if (flag == kFlagPrefix && j >= 0) {
                // Acquire: the prefix flag was seen; order the side-array read after it.
                __threadfence();
                mine = ld_relaxed_gpu_f64(prefix64 + j);
            } else if (flag == kFlagAggregate) {
                mine = double(__uint_as_float(value));
            }
        }
        exclusive += warp_sum(mine);
        if (prefix_mask != 0u || timed_out) break;
        win -= 32;
    }
    if (lane == 0) {
        const double inclusive = exclusive + double(aggregate);
        st_relaxed_gpu_f64(prefix64 + tile, inclusive);
        st_release_gpu(status + tile, pack_status(__float_as_uint(float(inclusive)), kFlagPrefix));
    }
    return exclusive;
}

// ---------------------------------------------------------------- predicates
//
// Elements are handled as raw 32-bit patterns.  Float "x != 0" is decided on
// the bits: every pattern except +0.0 and -0.0 compares unequal to zero under
// IEEE 754, NaNs and denormals included, and the bit test keeps that true
// whatever the compiler's denormal mode.
struct PredNonzeroInt {
    __device__ __forceinline__ bool operator()(uint32_t x) const { return x != 0u; }
};
struct PredNonzeroF32 {
    __device__ __forceinline__ bool operator()(uint32_t x) const { return (x & 0x7fffffffu) != 0u; }
};
struct PredOdd {
    __device__ __forceinline__ bool operator()(uint32_t x) const { return (x & 1u) != 0u; }
};
struct PredEven {
    __device__ __forceinline__ bool operator()(uint32_t x) const { return (x & 1u) == 0u; }
};
// Radix split: "bit b is clear" goes first.
struct PredBitClear {
    uint32_t bit;
    __device__ __forceinline__ bool operator()(uint32_t x) const { return ((x >> bit) & 1u) == 0u; }
};

// ---------------------------------------------------------------- tile geometry
//
// A tile is ROWS rows of THREADS x 4 consecutive elements.  Thread t owns the
// four elements [4t, 4t + 4) of every row, loaded as one 16-byte vector, so
// each warp load instruction covers 512 contiguous bytes.  Tile order is
// (row, warp, lane, item): a warp's 128 elements of one row form a "chunk",
// and chunk c = row * WARPS + warp is the c-th block of 128 in the tile.
template <int THREADS, int ROWS>
struct Tile {
    static constexpr int kThreads = THREADS;
    static constexpr int kRows = ROWS;
    static constexpr int kWarps = THREADS / 32;
    static constexpr int kRowElems = THREADS * 4;
    static constexpr int kElems = kRowElems * ROWS;
    static constexpr int kChunks = kWarps * ROWS;
    static_assert(THREADS % 32 == 0, "whole warps");
    static_assert(kChunks % 32 == 0, "chunk totals are scanned 32 at a time by one warp");
    static constexpr int kChunksPerLane = kChunks / 32;
};

// Loads the 4 elements at [idx, idx + 4) into v; elements at or past n get
// `fill`.  VEC: the pointer is 16-byte aligned and a full vector is one
// 128-bit load.
template <bool VEC>
__device__ __forceinline__ void load4(const uint32_t *__restrict__ in, uint32_t idx, uint32_t n,
                                      uint32_t fill, uint32_t (&v)[4])
{
    if (VEC && idx + 4u <= n) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(in + idx));
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = (idx + k < n) ? __ldcs(in + idx + k) : fill;
    }
}

template <bool VEC>
__device__ __forceinline__ void store4(uint32_t *__restrict__ out, uint32_t idx, uint32_t n,
                                       const uint32_t (&v)[4])
{
    if (VEC && idx + 4u <= n) {
        __stcs(reinterpret_cast<uint4 *>(out + idx), make_uint4(v[0], v[1], v[2], v[3]));
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (idx + k < n) __stcs(out + idx + k, v[k]);
    }
}

// Takes the next tile id for this CTA (one atomic, broadcast through smem).
__device__ __forceinline__ uint32_t claim_tile(uint8_t *ws, uint32_t *s_slot)
{
    if (threadIdx.x == 0) *s_slot = atomicAdd(hdr_u32(ws, kTileCtrOff), 1u);
    __syncthreads();
    return *s_slot;
}

// Exclusive scan, across warp 0, of the kChunks chunk totals in s_chunk
// (overwritten with the exclusive offsets).  Returns the tile total.
template <class TileT, class V>
__device__ __forceinline__ V scan_chunks_warp0(V *s_chunk)
{
    const int lane = threadIdx.x & 31;
    constexpr int K = TileT::kChunksPerLane;
    V c[K];
    V run = V(0);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        c[k] = s_chunk[lane * K + k];
        run += c[k];
    }
    V incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += y;
    }
    const V total = __shfl_sync(kFullMask, incl, 31);
    V excl = __shfl_up_sync(kFullMask, incl, 1);
    if (lane == 0) excl = V(0);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        s_chunk[lane * K + k] = excl;
        excl += c[k];
    }
    return total;
}


// Writes s[soff .. soff + len) to out[dst .. dst + len).  VEC: out is 16-byte
// aligned and soff - (dst & 3) is a multiple of 4, so the whole vectors of
// the run line up in both memories.
template <int THREADS, bool VEC>
__device__ __forceinline__ void store_run(uint32_t *__restrict__ out, uint32_t dst,
                                          const uint32_t *s, uint32_t soff, uint32_t len)
{
    if (len == 0u) return;
    if (VEC) {
        const uint32_t head = dst & 3u;
        const uint32_t g0 = dst - head;
        const uint32_t s0 = soff - head;
        const uint32_t span = head + len;
        const uint32_t nvec = (span + 3u) >> 2;
        for (uint32_t v = threadIdx.x; v < nvec; v += THREADS) {
            const uint32_t e = 4u * v;
            if (e >= head && e + 4u <= span) {
                const uint4 q = *reinterpret_cast<const uint4 *>(s + s0 + e);
                __stcs(reinterpret_cast<uint4 *>(out + g0 + e), q);
            } else {
#pragma unroll
                for (uint32_t k = 0; k < 4u; ++k)
                    if (e + k >= head && e + k < span) __stcs(out + g0 + e + k, s[s0 + e + k]);
            }
        }
    } else {
        for (uint32_t i = threadIdx.x; i < len; i += THREADS) __stcs(out + dst + i, s[soff + i]);
    }
}

// Per-row 4-bit keep masks of one thread's elements, and the thread's rank
// offsets: after this, rank of item k of row r within the tile's survivors is
// s_chunk[r * WARPS + warp] + lane_excl[r] + popc(mask[r] & ((1 << k) - 1)).
// Writes the chunk totals (packed scan, lane 31) into s_chunk.
template <class TT>
__device__ __forceinline__ void rank_masks(const uint32_t (&mask)[TT::kRows],
                                           uint32_t (&lane_excl)[TT::kRows], uint32_t *s_chunk)
{
    constexpr int ROWS = TT::kRows;
    constexpr int WORDS = (ROWS + 3) / 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t packed[WORDS];
#pragma unroll
    for (int w = 0; w < WORDS; ++w) packed[w] = 0u;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) packed[r / 4] |= uint32_t(__popc(mask[r])) << (8 * (r % 4));
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
        uint32_t incl = packed[w];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - packed[w];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = 4 * w + q;
            if (r < ROWS) {
                lane_excl[r] = (excl >> (8 * q)) & 0xffu;
                if (lane == 31) s_chunk[r * TT::kWarps + warp] = (incl >> (8 * q)) & 0xffu;
            }
        }
    }
}

}  // namespace gcd
