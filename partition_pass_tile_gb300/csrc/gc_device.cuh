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
// A persistent call clears its T status words inside its kernel, before a
// start barrier that every CTA passes before it publishes or reads one
// (bar_arrive / bar_wait below); the one-tile-per-CTA kernels have the tile
// counter and their status words cleared by one cudaMemsetAsync of
// [kTileCtrOff, 512 + 8 T) first.  Either way a status word is never read
// with contents from an earlier call.
constexpr uint32_t kHdrError = 0;        // u32: first device failure (gc_status), 0 = none
constexpr uint32_t kHdrErrorTile = 4;    // u32: tile whose wait gave up
constexpr uint32_t kHdrReduceCtr = 8;    // u32: CTAs finished in a count pre-pass (self-resetting)
constexpr uint32_t kHdrCountTrue = 12;   // u32: partition: elements the predicate keeps
constexpr uint32_t kHdrCountAcc = 16;    // u32: count pre-pass accumulator (reset by the last CTA)
constexpr uint32_t kHdrBarEpoch = 32;    // u32: start barriers completed (any value will do)
constexpr uint32_t kHdrBitAcc = 64;      // u32[32]: radix: keys with bit b set, accumulating
constexpr uint32_t kHdrBitZeros = 192;   // u32[32]: radix: keys with bit b clear
constexpr uint32_t kHdrBarArrive = 496;  // u32: CTAs arrived at a start barrier (self-resetting)
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

__device__ __forceinline__ uint32_t ld_relaxed_gpu_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// ---------------------------------------------------------------- start barrier
//
// A persistent call clears its own status words; this barrier keeps every
// publish and every read of a status word behind every CTA's share of the
// clear.  Thread 0 of each CTA reads the epoch word (bar_epoch) before its
// CTA arrives, and arrives (bar_arrive) once the whole CTA has cleared: one
// release add on the arrival counter.  The CTA whose add completes the count
// sets the counter back to 0 (so the zero-filled workspace and every
// completed barrier leave it at 0) and releases the epoch's next value; the
// others wait to acquire a changed epoch (bar_wait), the caller first waiting
// for its first tile's load so that the two latencies overlap.  A CTA
// barrier after that wait orders every thread's later accesses.  Every CTA
// reads the epoch before it arrives and the epoch changes only after the
// last arrival, so all of them read the same value.  The counter and the
// epoch sit in different 128-byte lines, so the waiting CTAs' polls of the
// one do not queue behind the adds on the other.
//
// The wait is bounded: past timeout_ns a CTA records GC_ERR_TIMEOUT (error
// tile kBarrierErrorTile), sets the counter's top bit so that no later call's
// barrier can complete on a count left over from this one (each times out
// and reports instead, until gc_query_device_status clears the counter), and
// carries on.
constexpr uint32_t kBarPoison = 0x80000000u;
constexpr uint32_t kBarrierErrorTile = 0xfffffffeu;

__device__ __forceinline__ uint32_t bar_epoch(uint8_t *ws)
{
    return ld_relaxed_gpu_u32(hdr_u32(ws, kHdrBarEpoch));
}

// Returns true if this CTA completed the barrier (nothing to wait for).
__device__ __forceinline__ bool bar_arrive(uint8_t *ws, uint32_t epoch)
{
    uint32_t *arrive = hdr_u32(ws, kHdrBarArrive);
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(arrive) : "memory");
    if (old != gridDim.x - 1u) return false;
    st_relaxed_gpu_u32(arrive, 0u);
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(hdr_u32(ws, kHdrBarEpoch)), "r"(epoch + 1u)
                 : "memory");
    return true;
}

__device__ __forceinline__ void bar_wait(uint8_t *ws, uint32_t epoch, uint64_t timeout_ns)
{
    const uint32_t *ep = hdr_u32(ws, kHdrBarEpoch);
    auto changed = [&]() {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ep) : "memory");
        return v != epoch;
    };
    if (changed()) return;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spins = 0; !changed(); ++spins) {
        if (spins >= 8) __nanosleep(64);
        if (global_timer_ns() - t0 > timeout_ns) {
            record_error(ws, kTimeoutCode, kBarrierErrorTile);
            atomicOr(hdr_u32(ws, kHdrBarArrive), kBarPoison);
            return;
        }
    }
}

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
// Parameterised predicate ("The CUDA Handbook, ch. 13": the compaction "is
// easily modified to evaluate more-complicated predicates"): a comparison
// with an operand in the dtype's own order (DT 0: int32 signed, 1: uint32
// unsigned, 2: float32 IEEE 754) or a test of the raw bits under a mask.
// Every element is mapped to an order-preserving unsigned key (int32: flip
// the sign bit; float32: flip the sign bit of positives and every bit of
// negatives, so keys ascend with the value and NaNs fall outside
// [key(-inf), key(+inf)]); each comparison then keeps one key interval
// [lo, lo + span] or, with invert, its complement.  The host turns the
// operator and operand into (lo, span, invert), treating -0.0 and +0.0 as
// equal and NaN operands as IEEE does, so each element costs a subtract, an
// unsigned compare and an xor.  A mask test keeps (x & mask) == value,
// inverted for "not equal".
template <int DT>
struct PredCmp {
    uint32_t lo;
    uint32_t span;
    uint32_t invert;
    uint32_t is_mask;
    uint32_t mask;
    uint32_t value;
    __device__ __forceinline__ bool operator()(uint32_t x) const
    {
        if (is_mask) return ((x & mask) == value) != (invert != 0u);
        uint32_t k = x;
        if (DT == 0) k = x ^ 0x80000000u;
        if (DT == 2) k = x ^ (uint32_t(int32_t(x) >> 31) | 0x80000000u);
        return ((k - lo) <= span) != (invert != 0u);
    }
};

// Radix split: "bit b is clear" goes first.
struct PredBitClear {
    uint32_t bit;
    __device__ __forceinline__ bool operator()(uint32_t x) const { return ((x >> bit) & 1u) == 0u; }
};

// Radix split on an order-preserving key of typed bits: key(x) = x ^
// (signfill(x) & neg) ^ flip ascends with the value, for int32 (neg 0, flip
// 2^31) and for float32 in IEEE 754 totalOrder (neg 2^31 - 1, flip 2^31: a
// negative pattern is inverted, a positive one gets its sign bit set).
// "Bit b of key(x) is clear" goes first; want is bit b of flip, so the key
// itself is never formed.
struct PredKeyBitClear {
    uint32_t bit, neg, want;
    __device__ __forceinline__ bool operator()(uint32_t x) const
    {
        const uint32_t sfill = uint32_t(int32_t(x) >> 31);
        return (((x ^ (sfill & neg)) >> bit) & 1u) == want;
    }
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
    static_assert(kChunks % 32 == 0 || (kChunks < 32 && 32 % kChunks == 0),
                  "chunk totals are scanned by one warp: a multiple of 32, or fewer");
    static constexpr int kChunksPerLane = kChunks >= 32 ? kChunks / 32 : 1;
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

// full_vec: the caller knows the vector is whole and 16-byte aligned.
template <bool VEC>
__device__ __forceinline__ void store4(uint32_t *__restrict__ out, uint32_t idx, uint32_t n,
                                       const uint32_t (&v)[4], bool full_vec = false)
{
    if (full_vec || (VEC && idx + 4u <= n)) {
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
    // with fewer than 32 chunks the lanes past the last one carry zeros
    constexpr bool kShort = TileT::kChunks < 32;
    V c[K];
    V run = V(0);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        c[k] = (!kShort || lane < TileT::kChunks) ? s_chunk[lane * K + k] : V(0);
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
        if (!kShort || lane < TileT::kChunks) s_chunk[lane * K + k] = excl;
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

// ---------------------------------------------------------------- CTA-wide look-back
//
// The same look-back with every thread of the CTA reading one predecessor, so
// one window covers THREADS tiles instead of 32.  Warps summarise their part
// of the window (is there a prefix, is anything missing before it, the sum up
// to it) in shared memory, and every thread combines the summaries in warp
// order, closest warp first.  The summaries are double-buffered by iteration
// parity, so one barrier per window suffices.  The time limit is decided from
// the warp leaders' clocks, OR-ed through the same summaries, so the whole
// CTA gives up in the same iteration.
struct LookbackSmem {
    uint32_t info[2][32];  // bit 0: prefix seen, bit 1: missing before it, bit 2: time is up
    uint32_t sum_u32[2][32];
    double sum_f64[2][32];
};

template <int THREADS, bool F32>
__device__ __forceinline__ void lookback_cta_impl(uint64_t *status, const double *prefix64,
                                                  uint32_t tile, uint8_t *ws, uint64_t timeout_ns,
                                                  LookbackSmem &sm, uint32_t &ex_u32,
                                                  double &ex_f64)
{
    constexpr int W = THREADS / 32;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int64_t win = int64_t(tile) - 1;
    int parity = 0;
    uint32_t spins = 0;
    uint64_t t_start = 0;
    ex_u32 = 0u;
    ex_f64 = 0.0;
    for (;;) {
        const int64_t j = win - t;
        uint32_t value = 0u, flag = kFlagPrefix;
        if (j >= 0) {
            const uint64_t w = ld_relaxed_gpu(status + j);
            value = uint32_t(w);
            flag = uint32_t(w >> 32);
        }
        const uint32_t pm = __ballot_sync(kFullMask, flag == kFlagPrefix);
        const uint32_t xm = __ballot_sync(kFullMask, flag == kFlagNone);
        const uint32_t use = lanes_up_to_first(pm);
        const bool mine = (use >> lane) & 1u;
        uint32_t su = 0u;
        double sd = 0.0;
        if (F32) {
            if (mine) {
                if (flag == kFlagPrefix && j >= 0) {
                    __threadfence();
                    sd = ld_relaxed_gpu_f64(prefix64 + j);
                } else if (flag == kFlagAggregate) {
                    sd = double(__uint_as_float(value));
                }
            }
            sd = warp_sum(sd);
        } else {
            su = warp_sum(mine && flag != kFlagNone ? value : 0u);
        }
        if (lane == 0) {
            const bool expired = spins > 0 && global_timer_ns() - t_start > timeout_ns;
            sm.info[parity][warp] = uint32_t(pm != 0u) | (uint32_t((xm & use) != 0u) << 1) |
                                    (uint32_t(expired) << 2);
            if (F32) sm.sum_f64[parity][warp] = sd; else sm.sum_u32[parity][warp] = su;
        }
        __syncthreads();
        uint32_t acc_u = 0u;
        double acc_d = 0.0;
        bool found = false, missing = false, expired = false;
#pragma unroll 1
        for (int w = 0; w < W; ++w) {
            const uint32_t info = sm.info[parity][w];
            expired |= (info >> 2) & 1u;
            if (!found) {
                missing |= (info >> 1) & 1u;
                if (F32) acc_d += sm.sum_f64[parity][w]; else acc_u += sm.sum_u32[parity][w];
                found = info & 1u;
            }
        }
        parity ^= 1;
        if (!missing || expired) {
            if (missing && t == 0) record_error(ws, kTimeoutCode, tile);
            ex_u32 += acc_u;
            ex_f64 += acc_d;
            if (found || missing) return;  // a prefix ends the walk; so does the time limit
            win -= THREADS;
            spins = 0;
            continue;
        }
        if (spins == 0) t_start = global_timer_ns();
        ++spins;
        __nanosleep(spins < 8 ? 20 : 100);
    }
}

// The tile's exclusive prefix and total, to every thread of the CTA.
// Chunk totals are in s_chunk (warp 0 scans them into offsets); warp 0 lane 0
// publishes the aggregate (or, for tile 0, the prefix) and, after the
// look-back, the inclusive prefix.  CTA_LOOKBACK picks the CTA-wide walk,
// otherwise warp 0 walks alone while the other warps wait at the barrier.
struct PrefixSmem {
    LookbackSmem lb;
    uint32_t res_u32[2];
    double res_f64;
    float agg_f32;
};

template <class TT, bool CTA_LOOKBACK>
__device__ __forceinline__ void resolve_prefix_u32(uint32_t *s_chunk, uint32_t tile, uint8_t *ws,
                                                   uint64_t timeout_ns, PrefixSmem &ps,
                                                   uint32_t &prefix, uint32_t &total)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *status = reinterpret_cast<uint64_t *>(ws + kStatusOff);
    if (!CTA_LOOKBACK) {
        if (warp == 0) {
            const uint32_t agg = scan_chunks_warp0<TT>(s_chunk);
            const uint32_t ex = lookback_u32(status, tile, agg, ws, timeout_ns);
            if (lane == 0) {
                ps.res_u32[0] = ex;
                ps.res_u32[1] = agg;
            }
        }
        __syncthreads();
        prefix = ps.res_u32[0];
        total = ps.res_u32[1];
        return;
    }
    if (warp == 0) {
        const uint32_t agg = scan_chunks_warp0<TT>(s_chunk);
        if (lane == 0) {
            ps.res_u32[1] = agg;
            st_relaxed_gpu(status + tile, pack_status(agg, tile == 0 ? kFlagPrefix : kFlagAggregate));
        }
    }
    __syncthreads();
    total = ps.res_u32[1];
    prefix = 0u;
    if (tile != 0) {
        double unused;
        lookback_cta_impl<TT::kThreads, false>(status, nullptr, tile, ws, timeout_ns, ps.lb, prefix,
                                               unused);
        if (threadIdx.x == 0) st_relaxed_gpu(status + tile, pack_status(prefix + total, kFlagPrefix));
    }
}

template <class TT, bool CTA_LOOKBACK>
__device__ __forceinline__ void resolve_prefix_f32(float *s_chunk, uint32_t tile, uint8_t *ws,
                                                   double *prefix64, uint64_t timeout_ns,
                                                   PrefixSmem &ps, double &prefix, float &total)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *status = reinterpret_cast<uint64_t *>(ws + kStatusOff);
    if (!CTA_LOOKBACK) {
        if (warp == 0) {
            const float agg = scan_chunks_warp0<TT>(s_chunk);
            const double ex = lookback_f32(status, prefix64, tile, agg, ws, timeout_ns);
            if (lane == 0) {
                ps.res_f64 = ex;
                ps.agg_f32 = agg;
            }
        }
        __syncthreads();
        prefix = ps.res_f64;
        total = ps.agg_f32;
        return;
    }
    if (warp == 0) {
        const float agg = scan_chunks_warp0<TT>(s_chunk);
        if (lane == 0) {
            ps.agg_f32 = agg;
            if (tile == 0) {
                st_relaxed_gpu_f64(prefix64, double(agg));
                st_release_gpu(status, pack_status(__float_as_uint(agg), kFlagPrefix));
            } else {
                st_relaxed_gpu(status + tile, pack_status(__float_as_uint(agg), kFlagAggregate));
            }
        }
    }
    __syncthreads();
    total = ps.agg_f32;
    prefix = 0.0;
    if (tile != 0) {
        uint32_t unused;
        lookback_cta_impl<TT::kThreads, true>(status, prefix64, tile, ws, timeout_ns, ps.lb, unused,
                                              prefix);
        if (threadIdx.x == 0) {
            const double inclusive = prefix + double(total);
            st_relaxed_gpu_f64(prefix64 + tile, inclusive);
            st_release_gpu(status + tile, pack_status(__float_as_uint(float(inclusive)), kFlagPrefix));
        }
    }
}

// ---------------------------------------------------------------- fixed-window prefix
//
// The persistent kernels own tiles round-robin: CTA c of G takes tiles c,
// c + G, c + 2G, ...  Each CTA keeps the inclusive prefix of its previous
// tile, R (the sum of every tile up to and including tile k - G), so the
// exclusive prefix of tile k is
//
//     prefix(k) = R + agg(k - G + 1) + ... + agg(k - 1)
//
// (for k < G: agg(0) + ... + agg(k - 1)).  Those G - 1 aggregates are
// published by the other CTAs as soon as they have reduced their tile, before
// they wait on anything, so one CTA-wide read of at most G - 1 status words
// gives the prefix: no tile ever waits on another tile's look-back, only on
// its aggregate.  This is the decoupled look-back of the CUDA Handbook's
// single-pass scan with the walk ending, always, at the CTA's own previous
// tile, whose inclusive prefix the CTA already holds.

// Publishes a tile's aggregate (one 64-bit store: value and flag together).
__device__ __forceinline__ void publish_aggregate(uint64_t *status, uint32_t tile, uint32_t bits)
{
    st_relaxed_gpu(status + tile, pack_status(bits, kFlagAggregate));
}

// Reads status word j until its aggregate is published (bounded wait: past
// timeout_ns it records GC_ERR_TIMEOUT and returns 0 for it).
__device__ __forceinline__ uint32_t await_aggregate(const uint64_t *status, uint32_t j, uint8_t *ws,
                                                    uint32_t tile, uint64_t timeout_ns)
{
    uint64_t w = ld_relaxed_gpu(status + j);
    if (uint32_t(w >> 32) != kFlagNone) return uint32_t(w);
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    for (;;) {
        __nanosleep(spins < 8 ? 32 : 128);
        ++spins;
        w = ld_relaxed_gpu(status + j);
        if (uint32_t(w >> 32) != kFlagNone) return uint32_t(w);
        if (global_timer_ns() - t0 > timeout_ns) {
            record_error(ws, kTimeoutCode, tile);
            return 0u;
        }
    }
}

// First tile of the window of tile k (the tiles after this CTA's previous one).
__device__ __forceinline__ uint32_t window_lo(uint32_t k)
{
    return k >= gridDim.x ? k - gridDim.x + 1u : 0u;
}

// ---------------------------------------------------------------- lagged window
//
// The window of a tile is read one iteration after its aggregates were
// published: a CTA reduces and publishes tile k, then finishes tile k - G
// (its previous one), whose window [k - 2G + 1, k - G) every CTA published a
// whole iteration earlier.  The loads of that window are issued before the
// reduction of tile k and consumed after it, so their latency overlaps the
// reduction.  kWinPerThread bounds the window: G - 1 <= THREADS * kWinPerThread.
#ifndef GC_WIN_PER_THREAD
#define GC_WIN_PER_THREAD 2
#endif
constexpr int kWinPerThread = GC_WIN_PER_THREAD;

struct WindowLoads {
    uint64_t w[kWinPerThread];
};

template <int THREADS>
__device__ __forceinline__ void window_issue(const uint64_t *status, uint32_t lo, uint32_t hi,
                                             WindowLoads &wl)
{
#pragma unroll
    for (int i = 0; i < kWinPerThread; ++i) {
        const uint32_t j = lo + threadIdx.x + uint32_t(i) * THREADS;
        wl.w[i] = j < hi ? ld_relaxed_gpu(status + j) : pack_status(0u, kFlagAggregate);
    }
}

// Completes the loads of window_issue (re-reading any word not yet
// published, bounded) and reduces them over the CTA; every thread gets the
// sum.  F32: the words hold float32 aggregates, summed in double.
template <int THREADS, bool F32>
__device__ __forceinline__ void window_finish(const uint64_t *status, uint32_t lo, uint32_t hi,
                                              WindowLoads &wl, uint8_t *ws, uint32_t tile,
                                              uint64_t timeout_ns, uint32_t *s_red_u,
                                              double *s_red_d, uint32_t &sum_u, double &sum_d)
{
    uint32_t su = 0u;
    double sd = 0.0;
#pragma unroll
    for (int i = 0; i < kWinPerThread; ++i) {
        const uint32_t j = lo + threadIdx.x + uint32_t(i) * THREADS;
        uint32_t v = uint32_t(wl.w[i]);
        if (j < hi && uint32_t(wl.w[i] >> 32) == kFlagNone) v = await_aggregate(status, j, ws, tile, timeout_ns);
        if (F32) sd += double(__uint_as_float(v)); else su += v;
    }
    if (F32) {
        sd = warp_sum(sd);
        if ((threadIdx.x & 31) == 0) s_red_d[threadIdx.x >> 5] = sd;
    } else {
        su = warp_sum(su);
        if ((threadIdx.x & 31) == 0) s_red_u[threadIdx.x >> 5] = su;
    }
    __syncthreads();
    sum_u = 0u;
    sum_d = 0.0;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) {
        if (F32) sum_d += s_red_d[w]; else sum_u += s_red_u[w];
    }
}

// Sum of one value over the CTA, to every thread.
template <int THREADS, class V>
__device__ __forceinline__ V block_sum_all(V v, V *s_red)
{
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    V t = V(0);
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) t += s_red[w];
    return t;
}

// ---------------------------------------------------------------- chunk offsets
// Every warp computes the exclusive scan of the tile's kChunks chunk totals
// (in s_chunk, chunk c = row * WARPS + warp) by itself and keeps the offsets
// of its own chunks, one per row, plus the tile total: one barrier (before
// the call) serves both the tile's reduction and its ranking.
struct NoTotalHook {
    template <class V>
    __device__ __forceinline__ void operator()(V) const {}
};

// on_total(total) runs as soon as the tile total is known, before the
// per-row offsets (a caller publishes it without waiting for them).
template <class TT, class V, class OnTotal = NoTotalHook>
__device__ __forceinline__ void chunk_offsets(const V *s_chunk, V (&off)[TT::kRows], V &total,
                                              const OnTotal &on_total = OnTotal{})
{
    constexpr int K = TT::kChunksPerLane;
    constexpr bool kShort = TT::kChunks < 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    V c[K];
    V run = V(0);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        c[k] = (!kShort || lane < TT::kChunks) ? s_chunk[lane * K + k] : V(0);
        run += c[k];
    }
    V incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(kFullMask, incl, 31);
    on_total(total);
    V e[K];
    e[0] = __shfl_up_sync(kFullMask, incl, 1);
    if (lane == 0) e[0] = V(0);
#pragma unroll
    for (int k = 1; k < K; ++k) e[k] = e[k - 1] + c[k - 1];
#pragma unroll
    for (int r = 0; r < TT::kRows; ++r) {
        const int ch = r * TT::kWarps + warp;  // warp-uniform
        V mine = e[0];
#pragma unroll
        for (int k = 1; k < K; ++k)
            if (ch % K == k) mine = e[k];
        off[r] = __shfl_sync(kFullMask, mine, ch / K);
    }
}

}  // namespace gcd
