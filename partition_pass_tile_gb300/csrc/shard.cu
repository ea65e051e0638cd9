// shard.cu -- the exchange step of a scan, select-if or partition split over
// P shards (one per GPU, or one after another on one GPU).
//
// An array cut into P contiguous shards is scanned, compacted or partitioned
// shard by shard once each shard knows what the shards before it contribute:
//
//   exclusive scan  carry(r)  = total(0) + ... + total(r - 1)
//   select-if       base(r)   = count(0) + ... + count(r - 1)
//   partition       kept(r)   = count(0) + ... + count(r - 1)
//                   rej(r)    = T + (n(0) + ... + n(r - 1)) - kept(r),
//                               T = count(0) + ... + count(P - 1)
//
// which is the exclusive scan of the P per-shard totals, the same "rank[i]
// is the number of survivors before i" and "i - rank[i]" arithmetic of
// "compaction.cu -- Day 33" (file header, scatterPartition), one level up.
// The P totals are all gathered to every rank (the only exchange); each rank
// then computes its own offsets here, on the device, so that the whole
// sequence pre-pass -> exchange -> offsets -> placed pass stays on one
// stream without a host synchronisation.
#include "gc_device.cuh"
#include "gc_internal.h"

namespace {

__global__ void shard_offsets_kernel(int op, int dt, const uint32_t *__restrict__ totals,
                                     uint32_t parts, uint32_t rank, uint64_t sizes_before,
                                     void *offsets)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (op == GC_OP_EXCLUSIVE_SCAN) {
        if (dt == GC_F32) {
            double acc = 0.0;
            for (uint32_t q = 0; q < rank; ++q) acc += double(__uint_as_float(totals[q]));
            *static_cast<uint32_t *>(offsets) = __float_as_uint(float(acc));
        } else {
            uint32_t acc = 0u;  // modulo 2^32, as the scan itself
            for (uint32_t q = 0; q < rank; ++q) acc += totals[q];
            *static_cast<uint32_t *>(offsets) = acc;
        }
        return;
    }
    uint64_t before = 0u, all = 0u;
    for (uint32_t q = 0; q < parts; ++q) {
        if (q < rank) before += totals[q];
        all += totals[q];
    }
    uint64_t *o = static_cast<uint64_t *>(offsets);
    o[0] = before;
    if (op == GC_OP_PARTITION) o[1] = all + (sizes_before - before);
}

}  // namespace

namespace gch {

cudaError_t launch_shard_offsets(gc_op op, gc_dtype dt, const uint32_t *totals, uint32_t parts,
                                 uint32_t rank, uint64_t sizes_before, void *offsets,
                                 cudaStream_t s)
{
    shard_offsets_kernel<<<1, 32, 0, s>>>(int(op), int(dt), totals, parts, rank, sizes_before,
                                          offsets);
    return cudaGetLastError();
}

}  // namespace gch
