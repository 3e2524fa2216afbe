// rsa_impl.cuh -- the fused reduce-scatter + AdamW + cast kernel ("K_RSA").
//
// One pass over the emulated ranks' blocks [begin, end) of the FlatParameter.
// For each element j it reads the N gradient values G_q[j] (rank order), the
// fp32 master / exp_avg / exp_avg_sq, and writes the three updated state
// values and the compute-dtype copy. Nothing else is read or written, so the
// algorithmic traffic per element is N*sizeof(grad) + 3*(4+4) + sizeof(out)
// bytes and the kernel is bound by HBM bandwidth (about 0.4 flop per byte).
//
// Sources: "Fully Sharded Data Parallel: faster AI training with fewer GPUs",
// "From all-reduce to sharded parameters" (reduce-scatter by rank block, local
// shard update); "Data Parallelism", "The Basic Protocol" (average by 1/N, then
// the Adam step); "fairseq ... FSDP 实战指南", "参数定义与底层实现"
// (--fp32-reduce-scatter) and "限制与兼容性说明" (pointwise optimizers);
// "FSDP (Fully Sharded Data Parallel)", "Mixed Precision and FSDP" (fp32
// master and state, bf16 compute copy).
//
// Variant with the fused all-gather (GATHER = true): every output element is
// also stored to the n_full gathered buffers, so the updated shards reach
// every emulated rank's full buffer in the same pass, without re-reading
// shard_out (which may then be omitted).
//
// Layout per thread and iteration: 8 consecutive elements. Each rank's 8
// bf16/fp16 gradients are one 16-byte load; master, m and v are two 16-byte
// loads each; the 8 outputs are one 16-byte store. All loads of an iteration
// are issued before any arithmetic so that each thread keeps N+6 16-byte
// requests in flight. Elements before the first 8-aligned index and after the
// last one (and every element when a base pointer is not 16-byte aligned) go
// through the scalar path, which performs the same operations in the same
// order.
//
// The launch code (grid sizing, dispatch over N and dtypes) is in
// rsa_launch.cuh.
#pragma once

#include "common.cuh"

namespace fsdp {
namespace rsa {

// Launch shape (compile-time tunables; the defaults are the measured best).
// Two builds of the kernel: state in HBM, 3 resident CTAs per SM (<= 80
// registers, no spills) and 8 consecutive elements per chunk; state in host
// memory, a 1-CTA launch bound and lane-interleaved chunks (SPLIT below),
// the layout the host link serves at full rate.
#ifndef FSDP_RSA_THREADS
#define FSDP_RSA_THREADS 256
#endif
#ifndef FSDP_RSA_MIN_BLOCKS
#define FSDP_RSA_MIN_BLOCKS 3
#endif
#ifndef FSDP_RSA_MIN_BLOCKS_HOST_STATE
#define FSDP_RSA_MIN_BLOCKS_HOST_STATE 1
#endif
constexpr int kThreads = FSDP_RSA_THREADS;
constexpr int kMinBlocks = FSDP_RSA_MIN_BLOCKS;
constexpr int kMinBlocksHostState = FSDP_RSA_MIN_BLOCKS_HOST_STATE;

// AdamW on one element; each operation is rounded on its own (no FMA), in the
// order of the documented definition.
__device__ __forceinline__ void adamw(float g, float &p, float &m, float &v, const AdamScalars &s) {
    p = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.b2s), s.eps);
    p = __fsub_rn(p, __fmul_rn(s.alpha, __fdiv_rn(m, denom)));
}

__device__ __forceinline__ uint32_t nonfinite(float g) { return isfinite(g) ? 0u : 1u; }

// The gathered buffers of a fused gather: n_full pointers at `full` (the
// per-unit kernel's own arguments, or one unit's descriptor in a batched
// launch); unused without GATHER.

// One element through the plain path.
template <int GD, int OD, bool GATHER>
__device__ __forceinline__ uint32_t scalar_elem(const RsaArgs &a, int world, int64_t j, void *const *full,
                                                int n_full) {
    float acc = Dtype<GD>::load(a.grads[0], j);
    for (int q = 1; q < world; ++q) acc = __fadd_rn(acc, Dtype<GD>::load(a.grads[q], j));
    const float g = __fmul_rn(acc, a.s.c);
    float p = a.master[j], m = a.m[j], v = a.v[j];
    adamw(g, p, m, v, a.s);
    a.master[j] = p;
    a.m[j] = m;
    a.v[j] = v;
    if (a.out != nullptr) Dtype<OD>::store(a.out, j, p);
    if constexpr (GATHER) {
        for (int d = 0; d < n_full; ++d) Dtype<OD>::store(full[d], j, p);
    }
    return nonfinite(g);
}

// Element layout of a thread's 8-element chunk: two 4-element halves at
// j_lo and j_hi. Consecutive (SPLIT false): j_hi = j_lo + 4, so each state
// buffer is read as two adjacent 16-byte words per thread. Lane-interleaved
// (SPLIT true, the build for state in host memory): in a warp's 256-element
// block lane l owns [4l, 4l + 4) and [128 + 4l, 128 + 4l + 4), so every
// warp-wide 16-byte state access covers 512 contiguous bytes; over the host
// link that layout moved twice the bytes of the adjacent-words one (a probe
// of the two patterns: 280-289 against 130-141 GB/s).

// Average, AdamW and cast of one 8-element chunk whose gradient sum is acc.
template <int OD, bool GATHER, bool SPLIT>
__device__ __forceinline__ uint32_t finish_chunk(const RsaArgs &a, int64_t j_lo, int64_t j_hi, const float *acc,
                                                 float4 p0, float4 p1, float4 m0, float4 m1,
                                                 float4 v0, float4 v1, void *const *full, int n_full) {
    float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t bad = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float g = __fmul_rn(acc[e], a.s.c);
        bad += nonfinite(g);
        adamw(g, p[e], m[e], v[e], a.s);
    }
    st_state(a.master + j_lo, make_float4(p[0], p[1], p[2], p[3]));
    st_state(a.master + j_hi, make_float4(p[4], p[5], p[6], p[7]));
    st_state(a.m + j_lo, make_float4(m[0], m[1], m[2], m[3]));
    st_state(a.m + j_hi, make_float4(m[4], m[5], m[6], m[7]));
    st_state(a.v + j_lo, make_float4(v[0], v[1], v[2], v[3]));
    st_state(a.v + j_hi, make_float4(v[4], v[5], v[6], v[7]));
    if constexpr (OD == FSDP_F32) {
        const float4 lo = make_float4(p[0], p[1], p[2], p[3]), hi = make_float4(p[4], p[5], p[6], p[7]);
        if (a.out != nullptr) {
            st_state(static_cast<float *>(a.out) + j_lo, lo);
            st_state(static_cast<float *>(a.out) + j_hi, hi);
        }
        if constexpr (GATHER) {
            for (int d = 0; d < n_full; ++d) {
                st_state(static_cast<float *>(full[d]) + j_lo, lo);
                st_state(static_cast<float *>(full[d]) + j_hi, hi);
            }
        }
    } else {
        const uint4 o = make_uint4(pack2<OD>(p[0], p[1]), pack2<OD>(p[2], p[3]),
                                   pack2<OD>(p[4], p[5]), pack2<OD>(p[6], p[7]));
        auto put = [&](void *base) {
            uint16_t *b = static_cast<uint16_t *>(base);
            if constexpr (SPLIT) {
                st_stream8(b + j_lo, make_uint2(o.x, o.y));
                st_stream8(b + j_hi, make_uint2(o.z, o.w));
            } else {
                st_stream(b + j_lo, o);
            }
        };
        if (a.out != nullptr) put(a.out);
        if constexpr (GATHER) {
            for (int d = 0; d < n_full; ++d) put(full[d]);
        }
    }
    return bad;
}

// Gradient registers of one 8-element chunk: one 16-byte word per rank for
// bf16/fp16, two for fp32.
template <int NW, int GD> struct GradRegs {
    static constexpr int kWords = GD == FSDP_F32 ? 2 : 1;
    uint4 w[NW > 0 ? NW : 1][kWords];
};

// One rank's gradients of a chunk (halves at j_lo and j_hi); bf16/fp16
// halves are packed into one 16-byte register word.
template <int GD, bool SPLIT>
__device__ __forceinline__ void load_grad8(const void *gq, int64_t j_lo, int64_t j_hi, uint4 *w) {
    if constexpr (GD == FSDP_F32) {
        w[0] = ld_stream(static_cast<const float *>(gq) + j_lo);
        w[1] = ld_stream(static_cast<const float *>(gq) + j_hi);
    } else if constexpr (SPLIT) {
        const uint2 lo = ld_stream8(static_cast<const uint16_t *>(gq) + j_lo);
        const uint2 hi = ld_stream8(static_cast<const uint16_t *>(gq) + j_hi);
        w[0] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    } else {
        w[0] = ld_stream(static_cast<const uint16_t *>(gq) + j_lo);
    }
}

// 8 consecutive elements from j0.
template <int GD>
__device__ __forceinline__ void load_grad8(const void *gq, int64_t j0, uint4 *w) {
    load_grad8<GD, false>(gq, j0, j0 + 4, w);
}

template <int GD> __device__ __forceinline__ void widen8(const uint4 *w, float *f) {
    if constexpr (GD == FSDP_F32) {
        const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(u[e]);
    } else {
        unpack8<GD>(w[0], f);
    }
}

template <int NW, int GD, int OD, bool GATHER, bool SPLIT>
__device__ __forceinline__ uint32_t vec_chunk(const RsaArgs &a, int world, int64_t j_lo, int64_t j_hi,
                                              void *const *full, int n_full) {
    float acc[8];
    if constexpr (NW > 0) {
        // every load of the chunk (N gradient words, then the state) is in
        // flight before the first add
        GradRegs<NW, GD> r;
#pragma unroll
        for (int q = 0; q < NW; ++q) load_grad8<GD, SPLIT>(a.grads[q], j_lo, j_hi, r.w[q]);
        const float4 p0 = ld_state(a.master + j_lo), p1 = ld_state(a.master + j_hi);
        const float4 m0 = ld_state(a.m + j_lo), m1 = ld_state(a.m + j_hi);
        const float4 v0 = ld_state(a.v + j_lo), v1 = ld_state(a.v + j_hi);
        widen8<GD>(r.w[0], acc);
#pragma unroll
        for (int q = 1; q < NW; ++q) {
            float f[8];
            widen8<GD>(r.w[q], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
        }
        return finish_chunk<OD, GATHER, SPLIT>(a, j_lo, j_hi, acc, p0, p1, m0, m1, v0, v1, full, n_full);
    } else {
        for (int q = 0; q < world; ++q) {
            uint4 w[GradRegs<1, GD>::kWords];
            load_grad8<GD, SPLIT>(a.grads[q], j_lo, j_hi, w);
            float f[8];
            widen8<GD>(w, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = q == 0 ? f[e] : __fadd_rn(acc[e], f[e]);
        }
        const float4 p0 = ld_state(a.master + j_lo), p1 = ld_state(a.master + j_hi);
        const float4 m0 = ld_state(a.m + j_lo), m1 = ld_state(a.m + j_hi);
        const float4 v0 = ld_state(a.v + j_lo), v1 = ld_state(a.v + j_hi);
        return finish_chunk<OD, GATHER, SPLIT>(a, j_lo, j_hi, acc, p0, p1, m0, m1, v0, v1, full, n_full);
    }
}

// Grid-stride over nchunks 8-element chunks starting at vbegin, then the
// scalar elements [begin, vbegin) and [vend, end). With nchunks = 0 and
// vbegin = vend = end every element takes the scalar path. With SPLIT the
// chunks are lane-interleaved within 256-element warp blocks (nchunks is a
// multiple of 32, and blockDim and the stride are multiples of 32, so the 32
// chunks k of a warp share one block).
template <int NW, int GD, int OD, bool GATHER, int MINB, bool SPLIT>
__global__ void __launch_bounds__(kThreads, MINB)
    rsa_kernel(const __grid_constant__ RsaArgs a, int64_t vbegin, int64_t nchunks, int64_t vend) {
    const int world = NW > 0 ? NW : a.world;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t bad = 0;
    for (int64_t k = tid; k < nchunks; k += stride) {
        int64_t j_lo, j_hi;
        if constexpr (SPLIT) {
            j_lo = vbegin + 256 * (k >> 5) + 4 * (k & 31);
            j_hi = j_lo + 128;
        } else {
            j_lo = vbegin + 8 * k;
            j_hi = j_lo + 4;
        }
        bad += vec_chunk<NW, GD, OD, GATHER, SPLIT>(a, world, j_lo, j_hi, a.full, a.n_full);
    }
    const int64_t nhead = vbegin - a.begin;
    const int64_t nrest = nhead + (a.end - vend);
    for (int64_t e = tid; e < nrest; e += stride) {
        const int64_t j = e < nhead ? a.begin + e : vend + (e - nhead);
        bad += scalar_elem<GD, OD, GATHER>(a, world, j, a.full, a.n_full);
    }
    if (a.nonfinite != nullptr) {
        const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
        if ((threadIdx.x & 31) == 0 && total) atomicAdd(a.nonfinite, total);
    }
}

}  // namespace rsa
}  // namespace fsdp
