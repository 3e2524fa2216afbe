// rsa_group.cu -- the batched fused update: one launch of the reduce-scatter
// + AdamW + cast over up to kGroupMax small units of one world size and one
// gradient / output dtype pair (group.cuh). Each CTA takes 256 of its unit's
// 8-element chunks, exactly as one CTA of the per-unit kernel does (the same
// loads, arithmetic and stores, through rsa_impl.cuh's chunk and element
// functions), and the unit's last CTA also takes the elements after the last
// whole chunk. The results are therefore bit-identical to the per-unit
// launches; only the launches, ramp-ups and tails per unit are saved.
#include "group.cuh"
#include "host.cuh"
#include "rsa_impl.cuh"

namespace fsdp {
namespace {

static_assert(rsa::kThreads == kGroupThreads, "the batched update's CTAs are sized for kGroupThreads threads");

// Launch bound: the per-unit kernel's 3 CTAs per SM (80 registers, no
// spills), except with fp32 gradients at N = 8, whose 16 gradient words per
// chunk plus the unit lookup spill 128 bytes per thread at that budget; 2 CTAs
// per SM (128 registers) cut that to 32-40 bytes.
template <int NW, int GD>
constexpr int group_min_blocks() {
    return (GD == FSDP_F32 && NW == 8) ? 2 : rsa::kMinBlocks;
}

template <int NW, int GD, int OD>
__global__ void __launch_bounds__(rsa::kThreads, group_min_blocks<NW, GD>())
    rsa_group_kernel(const __grid_constant__ RsaGroupArgs g) {
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
    const GroupUnit &U = g.u[lo];
    RsaArgs a;  // the fields the chunk and element functions read
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
    if (k < nchunks) bad += rsa::vec_chunk<NW, GD, OD, false, false>(a, NW, 8 * k, 8 * k + 4, nullptr, 0);
    if (local == U.ncta - 1) {
        for (int64_t j = 8 * nchunks + threadIdx.x; j < U.numel; j += blockDim.x)
            bad += rsa::scalar_elem<GD, OD, false>(a, NW, j, nullptr, 0);
    }
    if (g.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if ((threadIdx.x & 31) == 0 && total) atomicAdd(g.nonfinite, total);
    }
}

template <int NW, int GD, int OD>
fsdp_status launch_nw(const RsaGroupArgs &g, int64_t grid, cudaStream_t s) {
    rsa_group_kernel<NW, GD, OD><<<static_cast<unsigned>(grid), rsa::kThreads, 0, s>>>(g);
    return check_launch();
}

template <int GD, int OD>
fsdp_status launch_od(const RsaGroupArgs &g, int64_t grid, cudaStream_t s) {
    switch (g.world) {
        case 1: return launch_nw<1, GD, OD>(g, grid, s);
        case 2: return launch_nw<2, GD, OD>(g, grid, s);
        case 4: return launch_nw<4, GD, OD>(g, grid, s);
        case 8: return launch_nw<8, GD, OD>(g, grid, s);
        default: return FSDP_ERR_INVALID_ARG;
    }
}

template <int GD>
fsdp_status launch_gd(const RsaGroupArgs &g, int out_dtype, int64_t grid, cudaStream_t s) {
    switch (out_dtype) {
        case FSDP_BF16: return launch_od<GD, FSDP_BF16>(g, grid, s);
        case FSDP_F16: return launch_od<GD, FSDP_F16>(g, grid, s);
        case FSDP_F32: return launch_od<GD, FSDP_F32>(g, grid, s);
        default: return FSDP_ERR_UNSUPPORTED_DTYPE;
    }
}

}  // namespace

int32_t group_update_ctas(int64_t numel) {
    const int64_t per_cta = int64_t(8) * kGroupThreads;
    const int64_t n = (numel / 8 * 8 + per_cta - 1) / per_cta;
    return static_cast<int32_t>(n > 0 ? n : 1);
}

fsdp_status launch_rsa_group(const RsaGroupArgs &g, int grad_dtype, int out_dtype, int64_t grid, cudaStream_t s) {
    if (g.n < 1 || g.n > kGroupMax || grid < 1 || grid > 0x7fffffff) return FSDP_ERR_INVALID_ARG;
    switch (grad_dtype) {
        case FSDP_BF16: return launch_gd<FSDP_BF16>(g, out_dtype, grid, s);
        case FSDP_F16: return launch_gd<FSDP_F16>(g, out_dtype, grid, s);
        case FSDP_F32: return launch_gd<FSDP_F32>(g, out_dtype, grid, s);
        default: return FSDP_ERR_UNSUPPORTED_DTYPE;
    }
}

}  // namespace fsdp
