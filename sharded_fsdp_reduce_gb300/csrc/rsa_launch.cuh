// rsa_launch.cuh -- host launch code of the fused reduce-scatter + AdamW +
// cast kernel (rsa_impl.cuh): vector-path selection, grid sizing, dispatch
// over N, gradient dtype, output dtype and the fused all-gather.
//
// Grid. Not persistent: the grid is sized for about kChunksPerThread chunks
// per thread (at least one resident wave), so many more CTAs than fit on the
// GPU at once run in waves. Measured on the 70B and 13B units this is 7-8 %
// faster than a grid of exactly one resident wave striding over the whole
// range (e.g. 4.97 ms against 5.39-5.53 ms on the 70B unit); one chunk per
// thread with 3 CTAs per SM is 2.6 % faster again than two chunks with 2
// (4.994 against 5.127 ms in one process, bit-identical results).
// Builds: 3 resident CTAs per SM and consecutive chunks for state in HBM; a
// 1-CTA launch bound and lane-interleaved chunks (SPLIT) when the master
// lives in host memory (offload), the layout the host link serves at its
// full two-way rate (61.6 against 95 ms on the 70B unit).
#pragma once

#include "host.cuh"
#include "rsa_impl.cuh"

namespace fsdp {
namespace rsa {

#ifndef FSDP_RSA_CPT
#define FSDP_RSA_CPT 1
#endif
constexpr int kChunksPerThread = FSDP_RSA_CPT;

template <int NW, int GD, int OD, bool GATHER, int MINB, bool SPLIT>
fsdp_status launch_grid(const RsaArgs &a, cudaStream_t stream) {
    static std::atomic<int> occupancy{0};
    int blocks_per_sm = 1;
    const fsdp_status so =
        cached_occupancy(occupancy, rsa_kernel<NW, GD, OD, GATHER, MINB, SPLIT>, kThreads, 0, &blocks_per_sm);
    if (so != FSDP_OK) return so;
    bool vec = aligned(a.master, 16) && aligned(a.m, 16) && aligned(a.v, 16) && aligned(a.out, 16);
    for (int q = 0; q < a.world; ++q) vec = vec && aligned(a.grads[q], 16);
    for (int d = 0; d < a.n_full; ++d) vec = vec && aligned(a.full[d], 16);
    int64_t vbegin = a.end, vend = a.end, nchunks = 0;
    if (vec) {
        // the vector part: whole 8-element chunks from an 8-aligned start
        // (whole 256-element warp blocks with SPLIT)
        constexpr int64_t kUnit = SPLIT ? 256 : 8;
        vbegin = (a.begin + 7) / 8 * 8;
        vend = vbegin + (a.end > vbegin ? (a.end - vbegin) / kUnit * kUnit : 0);
        if (vend > vbegin) {
            nchunks = (vend - vbegin) / 8;
        } else {
            vbegin = vend = a.end;
        }
    }
    const int64_t items = nchunks + (vbegin - a.begin) + (a.end - vend);
    const int grid = grid_for(items, kThreads, kChunksPerThread, static_cast<int64_t>(sm_count()) * blocks_per_sm);
    rsa_kernel<NW, GD, OD, GATHER, MINB, SPLIT><<<grid, kThreads, 0, stream>>>(a, vbegin, nchunks, vend);
    return check_launch();
}

template <int NW, int GD, int OD, bool GATHER>
fsdp_status launch_typed(const RsaArgs &a, cudaStream_t stream) {
    return host_resident(a.master) ? launch_grid<NW, GD, OD, GATHER, kMinBlocksHostState, true>(a, stream)
                                   : launch_grid<NW, GD, OD, GATHER, kMinBlocks, false>(a, stream);
}

template <int GD, int OD, bool GATHER>
fsdp_status launch_world(const RsaArgs &a, cudaStream_t stream) {
    switch (a.world) {
        case 2: return launch_typed<2, GD, OD, GATHER>(a, stream);
        case 4: return launch_typed<4, GD, OD, GATHER>(a, stream);
        case 8: return launch_typed<8, GD, OD, GATHER>(a, stream);
        default: return launch_typed<0, GD, OD, GATHER>(a, stream);
    }
}

template <int GD, int OD>
fsdp_status launch_gather_flag(const RsaArgs &a, cudaStream_t stream) {
    return a.n_full > 0 ? launch_world<GD, OD, true>(a, stream) : launch_world<GD, OD, false>(a, stream);
}

template <int GD>
fsdp_status launch_grad(const RsaArgs &a, int out_dtype, cudaStream_t stream) {
    switch (out_dtype) {
        case FSDP_BF16: return launch_gather_flag<GD, FSDP_BF16>(a, stream);
        case FSDP_F16: return launch_gather_flag<GD, FSDP_F16>(a, stream);
        case FSDP_F32: return launch_gather_flag<GD, FSDP_F32>(a, stream);
        default: return FSDP_ERR_UNSUPPORTED_DTYPE;
    }
}

}  // namespace rsa
}  // namespace fsdp
