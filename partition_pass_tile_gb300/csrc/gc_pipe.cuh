// gc_pipe.cuh -- the load pipeline of the persistent tile kernels: tiles are
// copied from global into shared memory by the TMA unit (cp.async.bulk, one
// bulk copy per tile, completion signalled on an mbarrier), STAGES tiles
// ahead of the tile being computed on.
//
// Why: a tile kernel spends part of every tile waiting for its look-back
// (the predecessors' prefixes), and while it waits it issues no loads.  With
// the next STAGES - 1 tiles already in flight into shared memory the memory
// system stays busy through that wait, so the kernel can stream at the HBM
// rate with one or two CTAs per SM.
//
// Schedule: the grid is launched cooperatively (every CTA resident at once)
// and CTA c owns tiles c, c + G, c + 2G, ... (G = gridDim.x), which it
// computes in that order and prefetches STAGES ahead.  Tile k's look-back
// waits only on tiles below k, each owned by a resident CTA that reaches it
// before any later tile of its own, so the smallest unfinished tile is always
// being worked on: the look-back always makes progress.  Prefetching only a
// CTA's own future tiles keeps every claimed tile close to being published;
// tiles taken from a shared counter ahead of time would sit unpublished in
// one CTA's queue and stall every later tile's look-back.
//
// Protocol, per stage s (one mbarrier each, arrival count 1): thread 0 does
// arrive.expect_tx(bytes) and issues the bulk copy of the tile's first
// `bytes` bytes (the largest multiple of 16 the tile holds; the ragged tail
// of the last tile is read with plain loads by the consumers); all threads
// wait on the stage's phase parity, compute, and after a barrier thread 0
// re-arms the stage with the CTA's tile STAGES rounds later.
#pragma once

#include <cstdint>

#include "gc_device.cuh"

namespace gcd {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0u;
}

// Bulk copy of `bytes` (a multiple of 16) from global src (16-byte aligned)
// into shared dst (16-byte aligned); completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from shared src to global dst
// (both 16-byte aligned), in the current bulk group of this thread.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Until every bulk store this thread committed has read its shared source.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;");
}

// Until every bulk store this thread committed is complete.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shortest run worth a bulk store: below it the proxy fence and the wait for
// the bulk group before the stage is refilled cost more than the threads'
// own 128-bit stores.
constexpr uint32_t kBulkMinRun = 512u;

// Writes s[soff .. soff + len) to out[dst .. dst + len) when soff and dst
// agree modulo 4 elements (16 bytes) and out is 16-byte aligned: the
// aligned middle of the run goes out as one bulk copy issued and committed
// by lane 0 of warp `warp` (its own bulk group), the ragged head and tail
// (at most 3 elements each) as plain stores by lanes 1-3 and 5-7 of that
// warp.  The caller has made the run's shared-memory writes visible to the
// async proxy (fence.proxy.async by every writer, then a barrier), and the
// issuing lane waits for its group (bulk_wait_read_all) before the buffer is
// used again.  Runs issued by different warps go out in parallel.
template <int THREADS>
__device__ __forceinline__ void store_run_bulk(uint32_t *__restrict__ out, uint32_t dst,
                                               const uint32_t *s, uint32_t soff, uint32_t len,
                                               int warp)
{
    if (len == 0u || int(threadIdx.x >> 5) != warp) return;
    const uint32_t end = dst + len;
    const uint32_t a = min((dst + 3u) & ~3u, end);
    const uint32_t b = max(end & ~3u, a);
    const uint32_t lane = threadIdx.x & 31u;
    if (lane >= 1u && lane - 1u < a - dst) __stcs(out + dst + (lane - 1u), s[soff + (lane - 1u)]);
    if (lane >= 5u && lane - 5u < end - b)
        __stcs(out + b + (lane - 5u), s[soff + (b - dst) + (lane - 5u)]);
    if (lane == 0u && b > a) {
        bulk_store(out + a, s + soff + (a - dst), (b - a) * 4u);
        bulk_commit();
    }
}

// Warps whose lane 0 may issue bulk stores of a tile's runs.
constexpr int kBulkIssuers = 4;

// Every issuing lane: until its bulk stores have read their shared source.
__device__ __forceinline__ void bulk_issuers_wait_read()
{
    if ((threadIdx.x & 31u) == 0u && (threadIdx.x >> 5) < unsigned(kBulkIssuers)) bulk_wait_read_all();
}

// Every issuing lane: until its bulk stores are complete.
__device__ __forceinline__ void bulk_issuers_wait_all()
{
    if ((threadIdx.x & 31u) == 0u && (threadIdx.x >> 5) < unsigned(kBulkIssuers)) bulk_wait_all();
}

// Waits for a stage's phase.  The wait is bounded: past timeout_ns of device
// time it records GC_ERR_TIMEOUT and returns, and the caller carries on with
// whatever the buffer holds (every thread follows the same path afterwards,
// so no barrier is ever left unmatched).
__device__ __forceinline__ void mbar_wait(uint64_t *bar, uint32_t parity, uint8_t *ws,
                                          uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) {
            record_error(ws, kTimeoutCode, 0xffffffffu);
            return;
        }
    }
}

// Shared-memory layout of a pipelined kernel: STAGES stages, each holding one
// tile buffer per input array (ARRAYS of them: keys and payloads for the
// radix split), then the mbarriers.  Every buffer has 128 bytes of slack
// after the tile, room for the in-place compaction of select-if and
// partition, whose runs are shifted by up to 3 (each) elements to line up
// with 16-byte global addresses.
template <uint32_t TILE_BYTES, int STAGES, int ARRAYS = 1>
struct Pipe {
    static constexpr uint32_t kArrBytes = TILE_BYTES + 128u;
    static constexpr uint32_t kStageBytes = kArrBytes * ARRAYS;
    static constexpr uint32_t kBarOff = kStageBytes * STAGES;
    static constexpr uint32_t kBytes = kBarOff + 8u * STAGES;

    uint8_t *base;
    // Elements by which each input array's pointer lies past a 16-byte
    // boundary (0 .. 3).  A shifted array is copied from that boundary, one
    // vector longer, so element j of a tile sits at buf(s, a)[j + sh[a]].
    uint32_t sh[ARRAYS];

    // The stage buffer as written by the kernel (16-byte aligned: in-place
    // compaction and bulk stores).
    __device__ __forceinline__ uint32_t *buf(int s, int array = 0) const
    {
        return reinterpret_cast<uint32_t *>(base + s * kStageBytes + array * kArrBytes);
    }
    // The stage buffer as read: element j of the tile at rbuf(s, a)[j].
    __device__ __forceinline__ uint32_t *rbuf(int s, int array = 0) const
    {
        return buf(s, array) + sh[array];
    }
    __device__ __forceinline__ uint64_t *bar(int s) const
    {
        return reinterpret_cast<uint64_t *>(base + kBarOff) + s;
    }

    // Thread 0, once: set up the barriers.
    __device__ __forceinline__ void init() const
    {
        for (int s = 0; s < STAGES; ++s) mbar_init(bar(s), 1);
        fence_barrier_init();
    }

    // Thread 0: start copying tile `tile` (< the tile count) of each of the
    // ARRAYS arrays in `srcs` into stage s.
    __device__ __forceinline__ void issue(int s, const uint32_t *const (&srcs)[ARRAYS], uint32_t tile,
                                          uint32_t tile_elems, uint32_t n) const
    {
        const uint32_t first = tile * tile_elems;
        const uint32_t valid = min(tile_elems, n - first);
        // An aligned array: its whole vectors (the ragged end is read from
        // global memory).  A shifted one: from the 16-byte boundary below the
        // tile's first element up to the one above its last, every byte of it
        // in a 16-byte chunk that holds an element of the array.
        uint32_t bytes[ARRAYS], total = 0u;
#pragma unroll
        for (int a = 0; a < ARRAYS; ++a) {
            bytes[a] = sh[a] == 0u ? (valid & ~3u) * 4u : ((valid + sh[a] + 3u) & ~3u) * 4u;
            total += bytes[a];
        }
        if (total != 0u) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar(s), total);
#pragma unroll
            for (int a = 0; a < ARRAYS; ++a)
                if (bytes[a] != 0u) bulk_load(buf(s, a), srcs[a] + first - sh[a], bytes[a], bar(s));
        } else {
            mbar_arrive(bar(s));
        }
    }

    // Thread 0: the prologue, the first STAGES tiles of this CTA.
    __device__ __forceinline__ void prime(const uint32_t *const (&srcs)[ARRAYS], uint32_t tile_elems,
                                          uint32_t n, uint32_t num_tiles) const
    {
        for (int s = 0; s < STAGES; ++s) {
            const uint32_t t = blockIdx.x + uint32_t(s) * gridDim.x;
            if (t < num_tiles) issue(s, srcs, t, tile_elems, n);
        }
    }

    // Thread 0, after the barrier that ends the use of stage s by tile
    // `tile`: re-arm s with this CTA's tile STAGES rounds later.
    __device__ __forceinline__ void refill(int s, const uint32_t *const (&srcs)[ARRAYS], uint32_t tile,
                                           uint32_t tile_elems, uint32_t n, uint32_t num_tiles) const
    {
        const uint32_t t = tile + uint32_t(STAGES) * gridDim.x;
        if (t < num_tiles) issue(s, srcs, t, tile_elems, n);
    }
};

// Elements of tile `tile` that arrive in shared memory (the rest of a ragged
// last tile is read from global memory).
__device__ __forceinline__ uint32_t staged_elems(uint32_t tile, uint32_t tile_elems, uint32_t n)
{
    const uint32_t first = tile * tile_elems;
    return min(tile_elems, n - first) & ~3u;
}

// Vector of 4 elements at tile-local index li: from the stage buffer when it
// was copied there, otherwise from global memory (elements at or past n read
// as `fill`).  FULL: the whole tile is staged (every tile but a ragged last
// one), so no test is needed.
// SH: the kernel instance reads shifted stages (an input pointer that is not
// 16-byte aligned, sbuf = rbuf); its stage reads find the shift from sbuf's
// address, and an aligned kernel instance has no such test at all.
template <bool FULL = false, bool SH = false>
__device__ __forceinline__ void stage_load4(const uint32_t *sbuf, const uint32_t *__restrict__ gin,
                                            uint32_t base, uint32_t li, uint32_t staged, uint32_t n,
                                            uint32_t fill, uint32_t (&v)[4])
{
    // A shifted stage: two aligned vectors, and the four words of the element
    // vector.
    const uint32_t sh = SH ? (smem_addr(sbuf) >> 2) & 3u : 0u;
    if (SH && sh != 0u && (FULL || li + 4u <= staged)) {
        const uint32_t *al = sbuf - sh;
        const uint4 a = *reinterpret_cast<const uint4 *>(al + li);
        const uint4 b = *reinterpret_cast<const uint4 *>(al + li + 4u);
        if (sh == 1u) {
            v[0] = a.y; v[1] = a.z; v[2] = a.w; v[3] = b.x;
        } else if (sh == 2u) {
            v[0] = a.z; v[1] = a.w; v[2] = b.x; v[3] = b.y;
        } else {
            v[0] = a.w; v[1] = b.x; v[2] = b.y; v[3] = b.z;
        }
        return;
    }
    if (FULL || li + 4u <= staged) {
        const uint4 q = *reinterpret_cast<const uint4 *>(sbuf + li);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = (base + li + k < n) ? gin[base + li + k] : fill;
    }
}

}  // namespace gcd
