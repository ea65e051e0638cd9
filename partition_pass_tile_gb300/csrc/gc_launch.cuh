// gc_launch.cuh -- host side of the persistent pipelined kernels: one
// __global__ wrapper around pipeline_run and its cooperative launch.
#pragma once

#include <algorithm>

#include "gc_internal.h"
#include "gc_tiles.cuh"

namespace gcd {

#if GC_PIPE_MIN_BLOCKS > 0
#define GC_PIPE_BOUNDS(T) __launch_bounds__(T, GC_PIPE_MIN_BLOCKS)
#else
#define GC_PIPE_BOUNDS(T) __launch_bounds__(T)
#endif

template <int THREADS, int STAGES, class Op>
__global__ void GC_PIPE_BOUNDS(THREADS)
pipeline_kernel(Op op, uint32_t n, uint32_t num_tiles, uint8_t *ws, uint64_t timeout_ns,
                StatusPlan plan)
{
    extern __shared__ __align__(128) uint8_t smem[];
    pipeline_run<THREADS, STAGES>(op, smem, n, num_tiles, ws, timeout_ns, plan);
}

// Launches the cooperative persistent grid (as many CTAs as fit, at most one
// per tile), which clears its own tile status words unless o says they are
// clear already.  Returns the launch error; a refused cooperative launch (the
// device cannot hold the grid right now) lets the caller fall back to a
// one-tile-per-CTA kernel.
template <int THREADS, int STAGES, class Op>
cudaError_t launch_pipeline(const Op &op, uint32_t n, uint8_t *ws, cudaStream_t s,
                            const gch::LaunchOpts &o)
{
    uint32_t tiles = uint32_t(gch::ceil_div(n, Op::kTileElems));
    StatusPlan plan{o.status_region, o.reset_status ? 1u : 0u, o.clear_region, o.clear_words};
    uint64_t timeout_ns = o.timeout_ns;
    auto kernel = pipeline_kernel<THREADS, STAGES, Op>;
    constexpr uint32_t smem = Op::template PipeT<STAGES>::kBytes;
    int grid = gch::persistent_grid(reinterpret_cast<const void *>(kernel), THREADS, smem, tiles);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    grid = std::min(grid, pipeline_max_grid<THREADS>());
    Op op_copy = op;
    void *args[] = {&op_copy, &n, &tiles, &ws, &timeout_ns, &plan};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kernel), dim3(grid),
                                       dim3(THREADS), args, smem, s);
}

}  // namespace gcd
