// step_group.cuh -- the batched variant step: one launch of the fused
// reduce-scatter + optimizer step + cast (step_impl.cuh) over up to
// kGroupMax small units of one optimizer, world size and dtype set
// (group.cuh). Each CTA takes 256 of its unit's 8-element chunks through the
// per-unit kernel's chunk function, and the unit's last CTA also its
// elements after the last whole chunk, so the results are bit-identical to
// the per-unit launches. Instantiated once per optimizer
// (step_group_<optimizer>.cu).
#pragma once

#include "group.cuh"
#include "step_impl.cuh"

namespace fsdp {
namespace step {

static_assert(kThreads == kGroupThreads, "the batched update's CTAs are sized for kGroupThreads threads");

// Launch bound: the per-unit kernel's (3 CTAs per SM), except with fp32
// gradients at N = 8, whose 16 gradient words per chunk plus the unit lookup
// spill 48-128 bytes per thread at that budget; 2 CTAs per SM (128
// registers) there, which leaves 32-48 bytes of spills in some of those
// builds and none in SGD's.
template <int NW, int GD>
constexpr int group_min_blocks() {
    return (GD == FSDP_F32 && NW == 8) ? 2 : kMinBlocks;
}

template <int OPT, int NW, int GD, int OD, int SD>
__global__ void __launch_bounds__(kThreads, group_min_blocks<NW, GD>())
    step_group_kernel(const __grid_constant__ StepGroupArgs g) {
    // the unit of this CTA: the last one whose first CTA is at or before it
    const int64_t b = blockIdx.x;
    int lo = 0, hi = g.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g.u[mid].cta_begin <= b) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    const StepGroupUnit &U = g.u[lo];
    StepArgs a;  // the fields the chunk and element functions read
#pragma unroll
    for (int q = 0; q < NW; ++q) a.grads[q] = U.grads[q];
    a.param = U.param;
    a.s0 = U.s0;
    a.s1 = U.s1;
    a.out = U.out;
    a.nonfinite = nullptr;
    a.begin = 0;
    a.end = U.numel;
    a.k = g.k;
    a.world = NW;
    a.reduce_lowp = g.reduce_lowp;

    const int64_t local = b - U.cta_begin;
    const int64_t nchunks = U.numel / 8;
    const int64_t c = local * kThreads + threadIdx.x;
    uint32_t bad = 0;
    if (c < nchunks) bad += vec_chunk<OPT, NW, GD, OD, SD, false>(a, NW, 8 * c, 8 * c + 4);
    if (local == U.ncta - 1) {
        for (int64_t j = 8 * nchunks + threadIdx.x; j < U.numel; j += blockDim.x)
            bad += scalar_elem<OPT, GD, OD, SD>(a, NW, j);
    }
    if (g.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if ((threadIdx.x & 31) == 0 && total) atomicAdd(g.nonfinite, total);
    }
}

template <int OPT, int GD, int OD, int SD>
fsdp_status launch_group_world(const StepGroupArgs &g, int64_t grid, cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>(grid);
    switch (g.world) {
        case 1: step_group_kernel<OPT, 1, GD, OD, SD><<<blocks, kThreads, 0, s>>>(g); break;
        case 2: step_group_kernel<OPT, 2, GD, OD, SD><<<blocks, kThreads, 0, s>>>(g); break;
        case 4: step_group_kernel<OPT, 4, GD, OD, SD><<<blocks, kThreads, 0, s>>>(g); break;
        case 8: step_group_kernel<OPT, 8, GD, OD, SD><<<blocks, kThreads, 0, s>>>(g); break;
        default: return FSDP_ERR_INVALID_ARG;
    }
    return check_launch();
}

template <int OPT, int GD>
fsdp_status launch_group_dtypes(const StepGroupArgs &g, int out_dtype, int state_dtype, int64_t grid,
                                cudaStream_t s) {
    if (state_dtype == FSDP_F32) {
        switch (out_dtype) {
            case FSDP_BF16: return launch_group_world<OPT, GD, FSDP_BF16, FSDP_F32>(g, grid, s);
            case FSDP_F16: return launch_group_world<OPT, GD, FSDP_F16, FSDP_F32>(g, grid, s);
            default: return launch_group_world<OPT, GD, FSDP_F32, FSDP_F32>(g, grid, s);
        }
    }
    if (state_dtype == FSDP_BF16) return launch_group_world<OPT, GD, FSDP_BF16, FSDP_BF16>(g, grid, s);
    return launch_group_world<OPT, GD, FSDP_F16, FSDP_F16>(g, grid, s);
}

template <int OPT>
fsdp_status launch_group_opt(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype, int64_t grid,
                             cudaStream_t s) {
    if (g.n < 1 || g.n > kGroupMax || grid < 1 || grid > 0x7fffffff) return FSDP_ERR_INVALID_ARG;
    switch (grad_dtype) {
        case FSDP_BF16: return launch_group_dtypes<OPT, FSDP_BF16>(g, out_dtype, state_dtype, grid, s);
        case FSDP_F16: return launch_group_dtypes<OPT, FSDP_F16>(g, out_dtype, state_dtype, grid, s);
        default: return launch_group_dtypes<OPT, FSDP_F32>(g, out_dtype, state_dtype, grid, s);
    }
}

}  // namespace step
}  // namespace fsdp
