// rsa_group_fused.cu -- the batched fused update with the first all-gather
// fused in: one launch of the reduce-scatter + AdamW + cast over up to
// kFusedGroupMax small units of one world size and one gradient / output
// dtype pair, each updated element also stored to every one of its unit's
// gathered buffers (group.cuh). Each CTA takes 256 of its unit's 8-element
// chunks through rsa_impl.cuh's chunk and element functions with the fused
// gather, exactly as one CTA of the per-unit kernel with the gather fused
// does, and the unit's last CTA also takes the elements after the last whole
// chunk; the gathered buffers' pointers are read from the unit's descriptor
// in the kernel's parameter space. The results are therefore bit-identical
// to the per-unit launches of fsdp_reduce_scatter_adam_cast_gather.
#include "group.cuh"
#include "host.cuh"
#include "rsa_impl.cuh"

namespace fsdp {
namespace {

static_assert(rsa::kThreads == kGroupThreads, "the batched update's CTAs are sized for kGroupThreads threads");

// Launch bound: as the batched update without the gather (rsa_group.cu).
template <int NW, int GD>
constexpr int fused_group_min_blocks() {
    return (GD == FSDP_F32 && NW == 8) ? 2 : rsa::kMinBlocks;
}

template <int NW, int GD, int OD>
__global__ void __launch_bounds__(rsa::kThreads, fused_group_min_blocks<NW, GD>())
    rsa_fused_group_kernel(const __grid_constant__ RsaFusedGroupArgs g) {
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
    const FusedGroupUnit &U = g.u[lo];
    RsaArgs a;  // the fields the chunk and element functions read (not the gathered buffers)
#pragma unroll
    for (int q = 0; q < NW; ++q) a.grads[q] = U.grads[q];
    a.master = U.master;
    a.m = U.m;
    a.v = U.v;
    a.out = U.out;
    a.nonfinite = nullptr;
    a.begin = 0;
    a.end = U.numel;
    a.s = g.s;
    a.world = NW;
    a.n_full = 0;

    const int64_t local = b - U.cta_begin;
    const int64_t nchunks = U.numel / 8;
    const int64_t k = local * rsa::kThreads + threadIdx.x;
    uint32_t bad = 0;
    if (k < nchunks) bad += rsa::vec_chunk<NW, GD, OD, true, false>(a, NW, 8 * k, 8 * k + 4, U.full, U.n_full);
    if (local == U.ncta - 1) {
        for (int64_t j = 8 * nchunks + threadIdx.x; j < U.numel; j += blockDim.x)
            bad += rsa::scalar_elem<GD, OD, true>(a, NW, j, U.full, U.n_full);
    }
    if (g.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if ((threadIdx.x & 31) == 0 && total) atomicAdd(g.nonfinite, total);
    }
}

template <int NW, int GD, int OD>
fsdp_status launch_nw(const RsaFusedGroupArgs &g, int64_t grid, cudaStream_t s) {
    rsa_fused_group_kernel<NW, GD, OD><<<static_cast<unsigned>(grid), rsa::kThreads, 0, s>>>(g);
    return check_launch();
}

template <int GD, int OD>
fsdp_status launch_od(const RsaFusedGroupArgs &g, int64_t grid, cudaStream_t s) {
    switch (g.world) {
        case 1: return launch_nw<1, GD, OD>(g, grid, s);
        case 2: return launch_nw<2, GD, OD>(g, grid, s);
        case 4: return launch_nw<4, GD, OD>(g, grid, s);
        case 8: return launch_nw<8, GD, OD>(g, grid, s);
        default: return FSDP_ERR_INVALID_ARG;
    }
}

template <int GD>
fsdp_status launch_gd(const RsaFusedGroupArgs &g, int out_dtype, int64_t grid, cudaStream_t s) {
    switch (out_dtype) {
        case FSDP_BF16: return launch_od<GD, FSDP_BF16>(g, grid, s);
        case FSDP_F16: return launch_od<GD, FSDP_F16>(g, grid, s);
        case FSDP_F32: return launch_od<GD, FSDP_F32>(g, grid, s);
        default: return FSDP_ERR_UNSUPPORTED_DTYPE;
    }
}

}  // namespace

fsdp_status launch_rsa_fused_group(const RsaFusedGroupArgs &g, int grad_dtype, int out_dtype, int64_t grid,
                                   cudaStream_t s) {
    if (g.n < 1 || g.n > kFusedGroupMax || grid < 1 || grid > 0x7fffffff) return FSDP_ERR_INVALID_ARG;
    switch (grad_dtype) {
        case FSDP_BF16: return launch_gd<FSDP_BF16>(g, out_dtype, grid, s);
        case FSDP_F16: return launch_gd<FSDP_F16>(g, out_dtype, grid, s);
        case FSDP_F32: return launch_gd<FSDP_F32>(g, out_dtype, grid, s);
        default: return FSDP_ERR_UNSUPPORTED_DTYPE;
    }
}

}  // namespace fsdp
