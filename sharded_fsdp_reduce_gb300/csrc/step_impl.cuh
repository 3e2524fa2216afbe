// step_impl.cuh -- the fused reduce-scatter + optimizer step + cast for the
// variant steps: other pointwise optimizers (SGD with momentum, Adamax,
// Adadelta, and AdamW), a reduce-scatter summed in the gradient dtype, and a
// parameter + state kept in bf16/fp16 without an fp32 master.
//
// Sources: "fairseq ... FSDP 实战指南", "限制与兼容性说明" (FSDP works with
// the pointwise optimizers Adam, AdamW, Adadelta, Adamax, SGD) and
// "参数定义与底层实现" (--fp32-reduce-scatter is off by default: the reduction
// then runs in the gradient dtype); "Fully Sharded Data Parallel: faster AI
// training with fewer GPUs", "Harnessing FSDP's full power", item 4 (FP16
// master weights and FP16 reduce-scatter); "FSDP (Fully Sharded Data
// Parallel)", "Mixed Precision and FSDP" (pure bf16: params and Adam state
// in bf16, no fp32 master). The update rules are the textbook ones (the
// pages print none):
//   SGD (momentum mu = beta1): d = g + wd*p; b = d on the first step, else
//       b = mu*b + d; p = p - lr*b
//   Adamax: d = g + wd*p; m = b1*m + (1-b1)*d; u = max(b2*u, |d| + eps) (NaN
//       if either side is); p = p - alpha*(m/u), alpha = lr/(1-b1^t)
//   Adadelta (rho = beta1): d = g + wd*p; s = rho*s + (1-rho)*(d*d);
//       delta = (sqrt(a+eps)/sqrt(s+eps))*d; a = rho*a + (1-rho)*(delta*delta);
//       p = p - lr*delta
//   AdamW: as the main kernel (decoupled decay, bias-corrected, eps outside).
// Every operation is rounded to fp32 on its own. A gradient-dtype reduction
// rounds each partial sum to the gradient dtype. Low-precision state is
// widened, updated in fp32 and rounded (RNE) when stored; the parameter
// buffer is then the rank's compute-dtype shard itself.
//
// Same memory schedule as the main kernel: per thread and iteration 8
// consecutive elements, every load of the chunk issued before any
// arithmetic, a scalar path for heads, tails and unaligned pointers, and a
// non-persistent grid of about one chunk per thread; for state in host
// memory the chunks are lane-interleaved within 256-element warp blocks.
#pragma once

#include "host.cuh"
#include "rsa_impl.cuh"

namespace fsdp {
namespace step {

// Launch shape as the main kernel: one chunk per thread, not persistent;
// 3 resident CTAs per SM with the state in HBM (measured in the bench on the
// 70B unit against two chunks at 2 CTAs per SM: the bf16 reduction 5.31 ->
// 4.97 ms, Adadelta 4.98 -> 4.90 ms, the others within 1 %); with the
// parameter in host memory a 1-CTA launch bound and lane-interleaved chunks,
// as the fused AdamW kernel's host-state build.
#ifndef FSDP_STEP_CPT
#define FSDP_STEP_CPT 1
#endif
#ifndef FSDP_STEP_MIN_BLOCKS
#define FSDP_STEP_MIN_BLOCKS 3
#endif
#ifndef FSDP_STEP_MIN_BLOCKS_HOST_STATE
#define FSDP_STEP_MIN_BLOCKS_HOST_STATE 1
#endif
constexpr int kThreads = 256;
constexpr int kChunksPerThread = FSDP_STEP_CPT;
constexpr int kMinBlocks = FSDP_STEP_MIN_BLOCKS;
constexpr int kMinBlocksHostState = FSDP_STEP_MIN_BLOCKS_HOST_STATE;

template <int OPT> struct Opt;
template <> struct Opt<FSDP_OPT_ADAMW> { static constexpr int kStates = 2; };
template <> struct Opt<FSDP_OPT_SGD> { static constexpr int kStates = 1; };
template <> struct Opt<FSDP_OPT_ADAMAX> { static constexpr int kStates = 2; };
template <> struct Opt<FSDP_OPT_ADADELTA> { static constexpr int kStates = 2; };

template <int OPT>
__device__ __forceinline__ void update(float g, float &p, float &s0, float &s1, const StepScalars &k) {
    if constexpr (OPT == FSDP_OPT_ADAMW) {
        p = __fmul_rn(p, k.decay);
        s0 = __fadd_rn(__fmul_rn(k.beta1, s0), __fmul_rn(k.omb1, g));
        s1 = __fadd_rn(__fmul_rn(k.beta2, s1), __fmul_rn(k.omb2, __fmul_rn(g, g)));
        const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(s1), k.b2s), k.eps);
        p = __fsub_rn(p, __fmul_rn(k.alpha, __fdiv_rn(s0, denom)));
    } else if constexpr (OPT == FSDP_OPT_SGD) {
        const float d = __fadd_rn(g, __fmul_rn(k.wd, p));
        s0 = k.first_step ? d : __fadd_rn(__fmul_rn(k.beta1, s0), d);
        p = __fsub_rn(p, __fmul_rn(k.lr, s0));
    } else if constexpr (OPT == FSDP_OPT_ADAMAX) {
        const float d = __fadd_rn(g, __fmul_rn(k.wd, p));
        s0 = __fadd_rn(__fmul_rn(k.beta1, s0), __fmul_rn(k.omb1, d));
        const float a = __fmul_rn(k.beta2, s1), b = __fadd_rn(fabsf(d), k.eps);
        s1 = (a > b || a != a) ? a : b;
        p = __fsub_rn(p, __fmul_rn(k.alpha, __fdiv_rn(s0, s1)));
    } else {  // FSDP_OPT_ADADELTA
        const float d = __fadd_rn(g, __fmul_rn(k.wd, p));
        s0 = __fadd_rn(__fmul_rn(k.beta1, s0), __fmul_rn(k.omb1, __fmul_rn(d, d)));
        const float delta =
            __fmul_rn(__fdiv_rn(__fsqrt_rn(__fadd_rn(s1, k.eps)), __fsqrt_rn(__fadd_rn(s0, k.eps))), d);
        s1 = __fadd_rn(__fmul_rn(k.beta1, s1), __fmul_rn(k.omb1, __fmul_rn(delta, delta)));
        p = __fsub_rn(p, __fmul_rn(k.lr, delta));
    }
}

// x rounded to the gradient dtype and back (a partial sum of a reduction in
// that dtype).
template <int GD> __device__ __forceinline__ float round_to(float x) {
    if constexpr (GD == FSDP_BF16) return __bfloat162float(__float2bfloat16_rn(x));
    else if constexpr (GD == FSDP_F16) return __half2float(__float2half_rn(x));
    else return x;
}

// The 8 values of a chunk in a buffer of dtype DT <-> floats: halves at
// j_lo and j_hi (consecutive: j_hi = j_lo + 4; SPLIT: the host-state build's
// lane-interleaved chunks, as in the fused AdamW kernel).
template <int DT> struct Words { uint4 w[DT == FSDP_F32 ? 2 : 1]; };

__device__ __forceinline__ uint2 ld_state8(const void *p) {
    uint2 r;
    asm volatile("ld.global.cs.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

template <int DT, bool SPLIT>
__device__ __forceinline__ Words<DT> load_state8(const void *base, int64_t j_lo, int64_t j_hi) {
    Words<DT> r;
    if constexpr (DT == FSDP_F32) {
        const float *p = static_cast<const float *>(base);
        const float4 a = ld_state(p + j_lo), b = ld_state(p + j_hi);
        r.w[0] = make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z), __float_as_uint(a.w));
        r.w[1] = make_uint4(__float_as_uint(b.x), __float_as_uint(b.y), __float_as_uint(b.z), __float_as_uint(b.w));
    } else if constexpr (SPLIT) {
        const uint16_t *p = static_cast<const uint16_t *>(base);
        const uint2 lo = ld_state8(p + j_lo), hi = ld_state8(p + j_hi);
        r.w[0] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    } else {
        const float4 a = ld_state(reinterpret_cast<const float *>(static_cast<const uint16_t *>(base) + j_lo));
        r.w[0] = make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z), __float_as_uint(a.w));
    }
    return r;
}

template <int DT> __device__ __forceinline__ void widen(const Words<DT> &x, float *f) { rsa::widen8<DT>(x.w, f); }

template <int DT, bool SPLIT>
__device__ __forceinline__ void store8(void *base, int64_t j_lo, int64_t j_hi, const float *f) {
    if constexpr (DT == FSDP_F32) {
        float *p = static_cast<float *>(base);
        st_state(p + j_lo, make_float4(f[0], f[1], f[2], f[3]));
        st_state(p + j_hi, make_float4(f[4], f[5], f[6], f[7]));
    } else {
        const uint4 o = make_uint4(pack2<DT>(f[0], f[1]), pack2<DT>(f[2], f[3]), pack2<DT>(f[4], f[5]),
                                   pack2<DT>(f[6], f[7]));
        uint16_t *b = static_cast<uint16_t *>(base);
        if constexpr (SPLIT) {
            st_stream8(b + j_lo, make_uint2(o.x, o.y));
            st_stream8(b + j_hi, make_uint2(o.z, o.w));
        } else {
            st_stream(b + j_lo, o);
        }
    }
}

template <int OPT, int NW, int GD, int OD, int SD, bool SPLIT>
__device__ __forceinline__ uint32_t vec_chunk(const StepArgs &a, int world, int64_t j_lo, int64_t j_hi) {
    constexpr int K = Opt<OPT>::kStates;
    float acc[8];
    Words<SD> pw, s0w, s1w;
    if constexpr (NW > 0) {
        rsa::GradRegs<NW, GD> r;
#pragma unroll
        for (int q = 0; q < NW; ++q) rsa::load_grad8<GD, SPLIT>(a.grads[q], j_lo, j_hi, r.w[q]);
        pw = load_state8<SD, SPLIT>(a.param, j_lo, j_hi);
        s0w = load_state8<SD, SPLIT>(a.s0, j_lo, j_hi);
        if constexpr (K == 2) s1w = load_state8<SD, SPLIT>(a.s1, j_lo, j_hi);
        rsa::widen8<GD>(r.w[0], acc);
#pragma unroll
        for (int q = 1; q < NW; ++q) {
            float f[8];
            rsa::widen8<GD>(r.w[q], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[e] = __fadd_rn(acc[e], f[e]);
                if (a.reduce_lowp) acc[e] = round_to<GD>(acc[e]);
            }
        }
    } else {
        for (int q = 0; q < world; ++q) {
            uint4 w[rsa::GradRegs<1, GD>::kWords];
            rsa::load_grad8<GD, SPLIT>(a.grads[q], j_lo, j_hi, w);
            float f[8];
            rsa::widen8<GD>(w, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (q == 0) {
                    acc[e] = f[e];
                } else {
                    acc[e] = __fadd_rn(acc[e], f[e]);
                    if (a.reduce_lowp) acc[e] = round_to<GD>(acc[e]);
                }
            }
        }
        pw = load_state8<SD, SPLIT>(a.param, j_lo, j_hi);
        s0w = load_state8<SD, SPLIT>(a.s0, j_lo, j_hi);
        if constexpr (K == 2) s1w = load_state8<SD, SPLIT>(a.s1, j_lo, j_hi);
    }
    float p[8], s0[8], s1[8];
    widen<SD>(pw, p);
    widen<SD>(s0w, s0);
    if constexpr (K == 2) {
        widen<SD>(s1w, s1);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) s1[e] = 0.0f;
    }
    uint32_t bad = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float g = __fmul_rn(acc[e], a.k.c);
        bad += rsa::nonfinite(g);
        update<OPT>(g, p[e], s0[e], s1[e], a.k);
    }
    store8<SD, SPLIT>(a.param, j_lo, j_hi, p);
    store8<SD, SPLIT>(a.s0, j_lo, j_hi, s0);
    if constexpr (K == 2) store8<SD, SPLIT>(a.s1, j_lo, j_hi, s1);
    if constexpr (SD == FSDP_F32) store8<OD, SPLIT>(a.out, j_lo, j_hi, p);
    return bad;
}

template <int OPT, int GD, int OD, int SD>
__device__ __forceinline__ uint32_t scalar_elem(const StepArgs &a, int world, int64_t j) {
    constexpr int K = Opt<OPT>::kStates;
    float acc = Dtype<GD>::load(a.grads[0], j);
    for (int q = 1; q < world; ++q) {
        acc = __fadd_rn(acc, Dtype<GD>::load(a.grads[q], j));
        if (a.reduce_lowp) acc = round_to<GD>(acc);
    }
    const float g = __fmul_rn(acc, a.k.c);
    float p = Dtype<SD>::load(a.param, j), s0 = Dtype<SD>::load(a.s0, j);
    float s1 = K == 2 ? Dtype<SD>::load(a.s1, j) : 0.0f;
    update<OPT>(g, p, s0, s1, a.k);
    Dtype<SD>::store(a.param, j, p);
    Dtype<SD>::store(a.s0, j, s0);
    if constexpr (K == 2) Dtype<SD>::store(a.s1, j, s1);
    if constexpr (SD == FSDP_F32) Dtype<OD>::store(a.out, j, p);
    return rsa::nonfinite(g);
}

template <int OPT, int NW, int GD, int OD, int SD, int MINB, bool SPLIT>
__global__ void __launch_bounds__(kThreads, MINB)
    step_kernel(const __grid_constant__ StepArgs a, int64_t vbegin, int64_t nchunks, int64_t vend) {
    const int world = NW > 0 ? NW : a.world;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t bad = 0;
    for (int64_t c = tid; c < nchunks; c += stride) {
        int64_t j_lo, j_hi;
        if constexpr (SPLIT) {  // lane-interleaved 256-element warp blocks
            j_lo = vbegin + 256 * (c >> 5) + 4 * (c & 31);
            j_hi = j_lo + 128;
        } else {
            j_lo = vbegin + 8 * c;
            j_hi = j_lo + 4;
        }
        bad += vec_chunk<OPT, NW, GD, OD, SD, SPLIT>(a, world, j_lo, j_hi);
    }
    const int64_t nhead = vbegin - a.begin;
    const int64_t nrest = nhead + (a.end - vend);
    for (int64_t e = tid; e < nrest; e += stride) {
        const int64_t j = e < nhead ? a.begin + e : vend + (e - nhead);
        bad += scalar_elem<OPT, GD, OD, SD>(a, world, j);
    }
    if (a.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if ((threadIdx.x & 31) == 0 && total) atomicAdd(a.nonfinite, total);
    }
}

template <int OPT, int NW, int GD, int OD, int SD, int MINB, bool SPLIT>
fsdp_status launch_grid(const StepArgs &a, cudaStream_t stream) {
    static std::atomic<int> occupancy{0};
    int blocks_per_sm = 1;
    const fsdp_status so =
        cached_occupancy(occupancy, step_kernel<OPT, NW, GD, OD, SD, MINB, SPLIT>, kThreads, 0, &blocks_per_sm);
    if (so != FSDP_OK) return so;
    bool vec = aligned(a.param, 16) && aligned(a.s0, 16) && aligned(a.s1, 16) && aligned(a.out, 16);
    for (int q = 0; q < a.world; ++q) vec = vec && aligned(a.grads[q], 16);
    int64_t vbegin = a.end, vend = a.end, nchunks = 0;
    if (vec) {
        constexpr int64_t kUnit = SPLIT ? 256 : 8;  // whole chunks (whole warp blocks with SPLIT)
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
    step_kernel<OPT, NW, GD, OD, SD, MINB, SPLIT><<<grid, kThreads, 0, stream>>>(a, vbegin, nchunks, vend);
    return check_launch();
}

template <int OPT, int NW, int GD, int OD, int SD>
fsdp_status launch_typed(const StepArgs &a, cudaStream_t stream) {
    return host_resident(a.param) ? launch_grid<OPT, NW, GD, OD, SD, kMinBlocksHostState, true>(a, stream)
                                  : launch_grid<OPT, NW, GD, OD, SD, kMinBlocks, false>(a, stream);
}

template <int OPT, int GD, int OD, int SD>
fsdp_status launch_world(const StepArgs &a, cudaStream_t stream) {
    switch (a.world) {
        case 2: return launch_typed<OPT, 2, GD, OD, SD>(a, stream);
        case 8: return launch_typed<OPT, 8, GD, OD, SD>(a, stream);
        default: return launch_typed<OPT, 0, GD, OD, SD>(a, stream);
    }
}

// (state dtype, out dtype) pairs: fp32 master with any compute dtype, or a
// bf16/fp16 parameter that is its own shard.
template <int OPT, int GD>
fsdp_status launch_dtypes(const StepArgs &a, int out_dtype, int state_dtype, cudaStream_t stream) {
    if (state_dtype == FSDP_F32) {
        switch (out_dtype) {
            case FSDP_BF16: return launch_world<OPT, GD, FSDP_BF16, FSDP_F32>(a, stream);
            case FSDP_F16: return launch_world<OPT, GD, FSDP_F16, FSDP_F32>(a, stream);
            default: return launch_world<OPT, GD, FSDP_F32, FSDP_F32>(a, stream);
        }
    }
    if (state_dtype == FSDP_BF16) return launch_world<OPT, GD, FSDP_BF16, FSDP_BF16>(a, stream);
    return launch_world<OPT, GD, FSDP_F16, FSDP_F16>(a, stream);
}

template <int OPT>
fsdp_status launch_opt(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t stream) {
    switch (grad_dtype) {
        case FSDP_BF16: return launch_dtypes<OPT, FSDP_BF16>(a, out_dtype, state_dtype, stream);
        case FSDP_F16: return launch_dtypes<OPT, FSDP_F16>(a, out_dtype, state_dtype, stream);
        default: return launch_dtypes<OPT, FSDP_F32>(a, out_dtype, state_dtype, stream);
    }
}

}  // namespace step
}  // namespace fsdp
