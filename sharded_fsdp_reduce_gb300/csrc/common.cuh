// common.cuh -- device-side helpers of libfsdpreduce.so and the argument
// structs its kernels receive (not part of the ABI). Host plumbing lives in
// host.cuh.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fsdp.h"

namespace fsdp {

// ---------------------------------------------------------------- dtypes

template <int DT> struct Dtype;
template <> struct Dtype<FSDP_F32> {
    static constexpr int kSize = 4;
    __device__ __forceinline__ static float load(const void *base, int64_t j) {
        return static_cast<const float *>(base)[j];
    }
    __device__ __forceinline__ static void store(void *base, int64_t j, float x) {
        static_cast<float *>(base)[j] = x;
    }
};
template <> struct Dtype<FSDP_BF16> {
    static constexpr int kSize = 2;
    __device__ __forceinline__ static float load(const void *base, int64_t j) {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[j]);
    }
    __device__ __forceinline__ static void store(void *base, int64_t j, float x) {
        static_cast<__nv_bfloat16 *>(base)[j] = __float2bfloat16_rn(x);
    }
};
template <> struct Dtype<FSDP_F16> {
    static constexpr int kSize = 2;
    __device__ __forceinline__ static float load(const void *base, int64_t j) {
        return __half2float(static_cast<const __half *>(base)[j]);
    }
    __device__ __forceinline__ static void store(void *base, int64_t j, float x) {
        static_cast<__half *>(base)[j] = __float2half_rn(x);
    }
};

inline int dtype_size(int dt) { return dt == FSDP_F32 ? 4 : 2; }
inline bool dtype_valid(int dt) { return dt == FSDP_F32 || dt == FSDP_BF16 || dt == FSDP_F16; }

// ---------------------------------------------------------------- 16-byte streaming access
// Every byte of the step is touched once, so loads skip L1 allocation and
// stores are marked streaming (evict-first in L2).

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream8(void *p, const uint2 &v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Read-modify-write state (master, m, v) is rewritten by the same kernel, so
// it takes the coherent path, marked streaming.
__device__ __forceinline__ float4 ld_state(const float *p) {
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z),
                       __uint_as_float(r.w));
}

__device__ __forceinline__ void st_state(float *p, const float4 &v) {
    st_stream(p, make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                            __float_as_uint(v.w)));
}

// 8 packed 16-bit values <-> 8 floats
template <int DT> __device__ __forceinline__ void unpack8(const uint4 &u, float *f);
template <> __device__ __forceinline__ void unpack8<FSDP_BF16>(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
template <> __device__ __forceinline__ void unpack8<FSDP_F16>(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w[k]);
        float2 x = __half22float2(h);
        f[2 * k] = x.x;
        f[2 * k + 1] = x.y;
    }
}

template <int DT> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<FSDP_BF16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half, b -> high half
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<FSDP_F16>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- kernel arguments

struct AdamScalars {
    float c;         // 1 / (N * grad_scale)
    float decay;     // 1 - lr * wd
    float beta1, beta2;
    float omb1, omb2;  // 1 - beta1, 1 - beta2
    float alpha;     // lr / (1 - beta1^t)
    float b2s;       // sqrt(1 - beta2^t)
    float eps;
};

struct RsaArgs {
    const void *grads[FSDP_MAX_WORLD];
    float *master;
    float *m;
    float *v;
    void *out;
    uint32_t *nonfinite;
    int64_t begin;   // first flat element of the emulated ranks' blocks
    int64_t end;     // one past the last
    AdamScalars s;
    int world;
    // fused all-gather: also store every output element to full[0..n_full)
    void *full[FSDP_MAX_WORLD];
    int n_full;
};


// Scalars of the variant steps (computed in double on the host, rounded once).
struct StepScalars {
    float c;             // 1 / (N * grad_scale)
    float decay;         // AdamW: 1 - lr * wd
    float beta1, beta2;
    float omb1, omb2;    // 1 - beta1, 1 - beta2
    float alpha;         // AdamW, Adamax: lr / (1 - beta1^t)
    float b2s;           // AdamW: sqrt(1 - beta2^t)
    float eps;
    float lr;
    float wd;
    int first_step;      // SGD: t == 1
};

struct StepArgs {
    const void *grads[FSDP_MAX_WORLD];
    void *param;     // fp32 master, or the bf16/fp16 parameter shard
    void *s0;
    void *s1;        // NULL for SGD
    void *out;       // compute-dtype shard when the state is fp32, else NULL
    uint32_t *nonfinite;
    int64_t begin;
    int64_t end;
    StepScalars k;
    int world;
    int reduce_lowp; // sum in the gradient dtype
};


struct GatherArgs {
    const void *src;
    void *dst[FSDP_MAX_WORLD];
    int64_t nbytes;
    int n_dst;
    uint32_t *timeouts;  // the call's count of bounded waits that gave up (device, or NULL)
};


struct FlattenArgs {
    static constexpr int kBatch = 32;
    const void *src[kBatch];  // NULL: zero fill
    int64_t dst_byte_off[kBatch];
    int64_t nbytes[kBatch];
    void *dst;
    int count;
    int elem_size;
};


}  // namespace fsdp
