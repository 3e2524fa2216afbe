// rsa_tma.cuh -- the fused reduce-scatter + AdamW + cast with the operands
// staged through shared memory by the Tensor Memory Accelerator.
//
// Same arithmetic as rsa_impl.cuh (the same device function per element),
// different memory schedule: per tile of kTE consecutive elements, one
// producer thread issues 1-D bulk loads of the N gradient tiles and of the
// master / exp_avg / exp_avg_sq tiles into one shared-memory stage
// (completion counted in bytes on the stage's "full" mbarrier); the consumer
// warps read the stage, update it in place and write the compute-dtype tile
// next to it, make their writes visible to the async proxy and arrive on the
// stage's "done" mbarrier; the producer then bulk-stores the three state
// tiles and the output tile and, once those stores have read the stage,
// refills it with the tile kStages ahead (with the all-gather fused in, the
// output tile is also bulk-stored once per gathered buffer). Loads run
// kStages - 1 tiles ahead
// of the arithmetic, and each load or store is a single instruction for a
// whole multi-KB tile.
//
// Every mbarrier wait is bounded (about a second of SM clocks); a wait that
// gives up is counted (fsdp_take_wait_timeouts) and its warp stops.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace fsdp {
namespace rsa_tma {

#ifndef FSDP_RSA_TMA_STAGES
#define FSDP_RSA_TMA_STAGES 4
#endif
constexpr int kTE = 1024;                          // elements per tile
constexpr int kStages = FSDP_RSA_TMA_STAGES;
constexpr int kConsumerWarps = 8;                  // 256 consumer threads, 4 elements each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr long long kWaitLimitCycles = 1ll << 31;

// Per-stage layout: N gradient tiles, master, m, v, then the output tile.
template <int NW, int GD, int OD> struct Stage {
    static constexpr int kGrad = kTE * Dtype<GD>::kSize;
    static constexpr int kState = kTE * 4;
    static constexpr int kOut = kTE * Dtype<OD>::kSize;
    static constexpr int kP = NW * kGrad;
    static constexpr int kM = kP + kState;
    static constexpr int kV = kM + kState;
    static constexpr int kO = kV + kState;
    static constexpr int kBytes = kO + kOut;
    static constexpr int kLoadBytes = NW * kGrad + 3 * kState;
};

// Bounded waits that gave up in this kernel (one counter per translation unit
// that instantiates it).
static __device__ uint32_t g_rsa_tma_wait_timeouts;

static inline uint32_t take_wait_timeouts() {
    uint32_t n = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&n, g_rsa_tma_wait_timeouts, sizeof(n)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_rsa_tma_wait_timeouts, &zero, sizeof(zero));
    return n;
}

// 4 consecutive 16-bit values <-> floats
template <int DT> __device__ __forceinline__ void widen4(uint2 u, float *f) {
    const uint4 w = make_uint4(u.x, u.y, 0, 0);
    float t[8];
    unpack8<DT>(w, t);
    f[0] = t[0]; f[1] = t[1]; f[2] = t[2]; f[3] = t[3];
}

template <int NW, int GD, int OD>
__global__ void __launch_bounds__(kThreads, 1)
    rsa_tma_kernel(const __grid_constant__ RsaArgs a, int64_t first_elem, int64_t ntiles) {
    using L = Stage<NW, GD, OD>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t done[kStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            tma::mbar_init(&full[s], 1);
            tma::mbar_init(&done[s], kConsumerWarps);
        }
        tma::fence_mbar_init();
    }
    __syncthreads();
    const int64_t step = gridDim.x;
    const int64_t mine = ntiles > blockIdx.x ? (ntiles - blockIdx.x + step - 1) / step : 0;

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------------- producer
        if (lane != 0 || mine == 0) return;
        auto elem0 = [&](int64_t it) { return first_elem + (blockIdx.x + it * step) * kTE; };
        auto load = [&](int64_t it) {
            const int s = static_cast<int>(it % kStages);
            unsigned char *st = smem + s * L::kBytes;
            const int64_t j0 = elem0(it);
            tma::mbar_arrive_expect_tx(&full[s], L::kLoadBytes);
#pragma unroll
            for (int q = 0; q < NW; ++q)
                tma::bulk_load(st + q * L::kGrad, static_cast<const char *>(a.grads[q]) + j0 * Dtype<GD>::kSize,
                               L::kGrad, &full[s]);
            tma::bulk_load(st + L::kP, a.master + j0, L::kState, &full[s]);
            tma::bulk_load(st + L::kM, a.m + j0, L::kState, &full[s]);
            tma::bulk_load(st + L::kV, a.v + j0, L::kState, &full[s]);
        };
        for (int64_t it = 0; it < mine && it < kStages; ++it) load(it);
        for (int64_t it = 0; it < mine; ++it) {
            const int s = static_cast<int>(it % kStages);
            if (!tma::mbar_wait_bounded(&done[s], static_cast<uint32_t>((it / kStages) & 1), kWaitLimitCycles)) {
                atomicAdd(&g_rsa_tma_wait_timeouts, 1u);
                break;
            }
            unsigned char *st = smem + s * L::kBytes;
            const int64_t j0 = elem0(it);
            tma::bulk_store(a.master + j0, st + L::kP, L::kState);
            tma::bulk_store(a.m + j0, st + L::kM, L::kState);
            tma::bulk_store(a.v + j0, st + L::kV, L::kState);
            if (a.out != nullptr)
                tma::bulk_store(static_cast<char *>(a.out) + j0 * Dtype<OD>::kSize, st + L::kO, L::kOut);
            for (int d = 0; d < a.n_full; ++d)  // the fused all-gather: one more bulk store per buffer
                tma::bulk_store(static_cast<char *>(a.full[d]) + j0 * Dtype<OD>::kSize, st + L::kO, L::kOut);
            tma::bulk_commit();
            if (it >= 1 && it - 1 + kStages < mine) {
                tma::bulk_wait_read<1>();  // the previous tile's stores have read their stage
                load(it - 1 + kStages);
            }
        }
        tma::bulk_wait<0>();
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int c = threadIdx.x;  // 0..255: elements 4c .. 4c+3 of every tile
    uint32_t bad = 0;
    for (int64_t it = 0; it < mine; ++it) {
        const int s = static_cast<int>(it % kStages);
        if (!tma::mbar_wait_bounded(&full[s], static_cast<uint32_t>((it / kStages) & 1), kWaitLimitCycles)) {
            if (lane == 0) atomicAdd(&g_rsa_tma_wait_timeouts, 1u);
            break;
        }
        unsigned char *st = smem + s * L::kBytes;
        float acc[4];
        widen4<GD>(*reinterpret_cast<const uint2 *>(st + 8 * c), acc);
#pragma unroll
        for (int q = 1; q < NW; ++q) {
            float f[4];
            widen4<GD>(*reinterpret_cast<const uint2 *>(st + q * L::kGrad + 8 * c), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
        }
        float4 *pp = reinterpret_cast<float4 *>(st + L::kP) + c;
        float4 *mp = reinterpret_cast<float4 *>(st + L::kM) + c;
        float4 *vp = reinterpret_cast<float4 *>(st + L::kV) + c;
        float4 p4 = *pp, m4 = *mp, v4 = *vp;
        float p[4] = {p4.x, p4.y, p4.z, p4.w}, m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g = __fmul_rn(acc[e], a.s.c);
            bad += rsa::nonfinite(g);
            rsa::adamw(g, p[e], m[e], v[e], a.s);
        }
        *pp = make_float4(p[0], p[1], p[2], p[3]);
        *mp = make_float4(m[0], m[1], m[2], m[3]);
        *vp = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<uint2 *>(st + L::kO + 8 * c) = make_uint2(pack2<OD>(p[0], p[1]), pack2<OD>(p[2], p[3]));
        tma::fence_proxy_async_smem();  // these writes are read next by bulk stores
        __syncwarp();
        if (lane == 0) tma::mbar_arrive(&done[s]);
    }
    if (a.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if (lane == 0 && total) atomicAdd(a.nonfinite, total);
    }
}

template <int NW, int GD, int OD>
fsdp_status launch(const RsaArgs &a, int64_t first_elem, int64_t ntiles, cudaStream_t stream) {
    using L = Stage<NW, GD, OD>;
    static PerDeviceOnce configured;  // the opt-in is a per-device function attribute
    const int smem = kStages * L::kBytes;
    const int dev = current_device();
    if (!configured.is_done(dev)) {
        cudaError_t e = cudaFuncSetAttribute(rsa_tma_kernel<NW, GD, OD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem);
        if (e != cudaSuccess) return cuda_status(e);
        configured.mark(dev);
    }
    const int64_t cap = sm_count();
    const int grid = static_cast<int>(ntiles < cap ? ntiles : cap);
    rsa_tma_kernel<NW, GD, OD><<<grid, kThreads, smem, stream>>>(a, first_elem, ntiles);
    return check_launch();
}

}  // namespace rsa_tma
}  // namespace fsdp
