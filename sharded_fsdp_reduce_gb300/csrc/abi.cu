// abi.cu -- the extern "C" entry points of libfsdpreduce.so (declared in
// include/fsdp.h): argument validation, the per-step scalars, and dispatch to
// the kernels. Every check runs on the host before anything is enqueued.
#include <cuda.h>  // the driver's pointer-attribute types: the call itself goes through the runtime's lookup
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <iterator>
#include <memory>
#include <new>
#include <vector>

#include "group.cuh"
#include "host.cuh"

// The library's exported symbols: the C ABI of include/fsdp.h and nothing else
// (everything else is built with hidden visibility).
#define FSDP_API __attribute__((visibility("default")))

namespace fsdp {

namespace {
thread_local int g_last_cuda_error = 0;
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // per device ordinal, 0 = not queried
}  // namespace

fsdp_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FSDP_OK;
    g_last_cuda_error = static_cast<int>(e);
    return FSDP_ERR_CUDA;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    const int slot = dev < kMaxDevices ? dev : 0;  // beyond 64 devices: slot 0's count (same part assumed)
    int n = g_sm_count[slot].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sm_count[slot].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

// cuPointerGetAttributes, found once through the runtime's driver entry-point
// lookup (the library links no driver library of its own); null if the
// lookup fails.
using PointerAttributesFn = CUresult (*)(unsigned int, CUpointer_attribute *, void **, CUdeviceptr);
PointerAttributesFn pointer_attributes_fn() {
    static const PointerAttributesFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f) {
            (void)cudaGetLastError();
            return static_cast<PointerAttributesFn>(nullptr);
        }
        return reinterpret_cast<PointerAttributesFn>(f);
    }();
    return fn;
}

}  // namespace

// One driver query gives a pointer's memory type, whether it is managed and
// the address range of its allocation; where that query is not available
// (no driver entry point, no current context) the runtime's query answers
// for this pointer alone. The classes match host_resident(): host memory
// (page-locked) and addresses the runtime does not know are host; device
// and managed memory are not.
bool ResidencyMemo::host_resident(const void *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    auto next = device_.upper_bound(a);  // the first kept allocation that starts after p
    if (next != device_.begin() && a < std::prev(next)->second) return false;
    if (const PointerAttributesFn fn = pointer_attributes_fn()) {
        // each value in a zeroed 8-byte word, whatever width the driver writes
        uint64_t type = 0, managed = 0, start = 0, size = 0;
        CUpointer_attribute attrs[4] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_IS_MANAGED,
                                        CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, CU_POINTER_ATTRIBUTE_RANGE_SIZE};
        void *data[4] = {&type, &managed, &start, &size};
        if (fn(4, attrs, data, static_cast<CUdeviceptr>(a)) == CUDA_SUCCESS) {
            if (managed != 0) return false;
            if (type == CU_MEMORYTYPE_DEVICE) {
                if (size > 0 && start <= a && a - start < size) {
                    try {
                        device_[start] = start + size;
                    } catch (...) {
                        // out of host memory: the range is not kept, and later pointers are queried
                    }
                }
                return false;
            }
            return type == CU_MEMORYTYPE_HOST || type == 0;
        }
    }
    return fsdp::host_resident(p);
}

namespace {

// Per-step scalars from the hyperparameters: computed in double, rounded
// once to float (the kernel then works in fp32 only).
AdamScalars make_scalars(const fsdp_adamw_hparams &h, int world) {
    const double t = static_cast<double>(h.step);
    AdamScalars s;
    s.c = static_cast<float>(1.0 / (static_cast<double>(world) * static_cast<double>(h.grad_scale)));
    s.decay = static_cast<float>(1.0 - static_cast<double>(h.lr) * static_cast<double>(h.weight_decay));
    s.beta1 = h.beta1;
    s.beta2 = h.beta2;
    s.omb1 = static_cast<float>(1.0 - static_cast<double>(h.beta1));
    s.omb2 = static_cast<float>(1.0 - static_cast<double>(h.beta2));
    s.alpha = static_cast<float>(static_cast<double>(h.lr) / (1.0 - pow(static_cast<double>(h.beta1), t)));
    s.b2s = static_cast<float>(sqrt(1.0 - pow(static_cast<double>(h.beta2), t)));
    s.eps = h.eps;
    return s;
}

bool mul_overflows(int64_t a, int64_t b) { return a != 0 && b > INT64_MAX / a; }

// Run the body of an entry point that allocates host memory for the
// library's own bookkeeping (the per-unit plans, batches and captured-step
// records): running out of it is reported as FSDP_ERR_HOST_MEMORY, never as
// an exception leaving the C ABI.
template <class Body>
fsdp_status guarded(Body &&body) noexcept {
    try {
        return body();
    } catch (...) {
        return FSDP_ERR_HOST_MEMORY;
    }
}

StepScalars make_step_scalars(const fsdp_step_config &c, int world) {
    const double t = static_cast<double>(c.step);
    StepScalars k;
    k.c = static_cast<float>(1.0 / (static_cast<double>(world) * static_cast<double>(c.grad_scale)));
    k.decay = static_cast<float>(1.0 - static_cast<double>(c.lr) * static_cast<double>(c.weight_decay));
    k.beta1 = c.beta1;
    k.beta2 = c.beta2;
    k.omb1 = static_cast<float>(1.0 - static_cast<double>(c.beta1));
    k.omb2 = static_cast<float>(1.0 - static_cast<double>(c.beta2));
    k.alpha = static_cast<float>(static_cast<double>(c.lr) / (1.0 - pow(static_cast<double>(c.beta1), t)));
    k.b2s = static_cast<float>(sqrt(1.0 - pow(static_cast<double>(c.beta2), t)));
    k.eps = c.eps;
    k.lr = c.lr;
    k.wd = c.weight_decay;
    k.first_step = c.step == 1 ? 1 : 0;
    return k;
}

}  // namespace
}  // namespace fsdp

using namespace fsdp;

extern "C" {

FSDP_API int64_t fsdp_padded_numel(int64_t numel, int world) {
    if (numel < 0 || world < 1) return -1;
    int64_t shards = numel / world;
    if (shards * world < numel) shards += 1;
    return shards * world;
}

FSDP_API fsdp_status fsdp_unflatten_views(const int64_t *shapes, const int32_t *ndims, int n_tensors, int world,
                                 fsdp_view *views_out, int64_t *padded_numel_out) {
    if (n_tensors < 0 || world < 1 || !padded_numel_out) return FSDP_ERR_INVALID_ARG;
    if (n_tensors > 0 && (!ndims || !views_out)) return FSDP_ERR_INVALID_ARG;
    int64_t at = 0;
    for (int k = 0; k < n_tensors; ++k) {
        if (ndims[k] < 0 || ndims[k] > FSDP_MAX_NDIM) return FSDP_ERR_INVALID_ARG;
        if (ndims[k] > 0 && !shapes) return FSDP_ERR_INVALID_ARG;
    }
    int64_t offset = 0;
    for (int k = 0; k < n_tensors; ++k) {
        fsdp_view v;
        memset(&v, 0, sizeof(v));
        v.ndim = ndims[k];
        int64_t numel = 1;
        for (int d = 0; d < ndims[k]; ++d) {
            const int64_t dim = shapes[at + d];
            if (dim < 0 || mul_overflows(numel, dim)) return FSDP_ERR_INVALID_ARG;
            v.shape[d] = dim;
            numel *= dim;
        }
        at += ndims[k];
        if (offset > INT64_MAX - numel) return FSDP_ERR_INVALID_ARG;
        v.offset = offset;
        v.numel = numel;
        offset += numel;
        views_out[k] = v;
    }
    const int64_t padded = fsdp_padded_numel(offset, world);
    if (padded < 0) return FSDP_ERR_INVALID_ARG;
    *padded_numel_out = padded;
    return FSDP_OK;
}

FSDP_API fsdp_status fsdp_flatten_pad(const void *const *srcs, const int64_t *numels, int n_tensors, fsdp_dtype dtype,
                             int world, void *dst_flat, int64_t dst_numel, fsdp_view *views_out,
                             void *stream) {
    if (!dtype_valid(dtype)) return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (n_tensors < 0 || world < 1 || dst_numel < 0) return FSDP_ERR_INVALID_ARG;
    if (n_tensors > 0 && (!srcs || !numels)) return FSDP_ERR_INVALID_ARG;
    const size_t es = static_cast<size_t>(dtype_size(dtype));
    int64_t total = 0;
    for (int k = 0; k < n_tensors; ++k) {
        if (numels[k] < 0 || total > INT64_MAX - numels[k]) return FSDP_ERR_INVALID_ARG;
        if (numels[k] > 0 && !srcs[k]) return FSDP_ERR_INVALID_ARG;
        total += numels[k];
    }
    const int64_t padded = fsdp_padded_numel(total, world);
    if (padded != dst_numel || mul_overflows(padded, static_cast<int64_t>(es))) return FSDP_ERR_INVALID_ARG;
    if (padded > 0 && !dst_flat) return FSDP_ERR_INVALID_ARG;
    if (dst_flat && !aligned(dst_flat, es)) return FSDP_ERR_ALIGNMENT;
    for (int k = 0; k < n_tensors; ++k) {
        if (numels[k] == 0) continue;
        if (!aligned(srcs[k], es)) return FSDP_ERR_ALIGNMENT;
        if (overlaps(srcs[k], numels[k] * es, dst_flat, padded * es)) return FSDP_ERR_INVALID_ARG;
    }
    if (views_out) {
        int64_t off = 0;
        for (int k = 0; k < n_tensors; ++k) {
            fsdp_view v;
            memset(&v, 0, sizeof(v));
            v.ndim = 1;
            v.shape[0] = numels[k];
            v.offset = off;
            v.numel = numels[k];
            views_out[k] = v;
            off += numels[k];
        }
    }
    // segments: each tensor, then the zero padding
    FlattenArgs a;
    memset(&a, 0, sizeof(a));
    a.dst = dst_flat;
    a.elem_size = static_cast<int>(es);
    int64_t off = 0;
    for (int k = 0; k <= n_tensors; ++k) {
        const bool pad = k == n_tensors;
        const int64_t n = pad ? padded - total : numels[k];
        if (n > 0) {
            a.src[a.count] = pad ? nullptr : srcs[k];
            a.dst_byte_off[a.count] = off * static_cast<int64_t>(es);
            a.nbytes[a.count] = n * static_cast<int64_t>(es);
            a.count += 1;
        }
        off += n;
        if (a.count == FlattenArgs::kBatch || (pad && a.count > 0)) {
            const fsdp_status st = launch_flatten(a, static_cast<cudaStream_t>(stream));
            if (st != FSDP_OK) return st;
            a.count = 0;
        }
    }
    return FSDP_OK;
}

}  // extern "C"

namespace {

// Validation shared by the fused update with and without the fused all-gather
// (full_bufs / n_dst; shard_out may then be NULL) and by the multi-unit step:
// fills the kernel's arguments, or sets `empty` when the rank range holds no
// element. Nothing is enqueued.
fsdp_status prepare_rsa(const void *const *grads, fsdp_dtype grad_dtype, int world, int64_t padded_numel,
                        float *master, float *exp_avg, float *exp_avg_sq, void *shard_out, fsdp_dtype out_dtype,
                        void *const *full_bufs, int n_dst, const fsdp_adamw_hparams *hp, int rank_begin,
                        int rank_end, uint32_t *nonfinite_count, RsaArgs &a, bool &empty) {
    empty = false;
    if (!dtype_valid(grad_dtype) || !dtype_valid(out_dtype)) return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (world < 1 || world > FSDP_MAX_WORLD || !grads || !hp) return FSDP_ERR_INVALID_ARG;
    if (padded_numel < 0 || padded_numel % world != 0) return FSDP_ERR_INVALID_ARG;
    if (rank_begin < 0 || rank_begin > rank_end || rank_end > world) return FSDP_ERR_INVALID_ARG;
    if (hp->step < 1 || !(hp->grad_scale > 0.0f) || !isfinite(hp->grad_scale)) return FSDP_ERR_INVALID_ARG;
    if (n_dst < 0 || n_dst > FSDP_MAX_WORLD || (n_dst > 0 && !full_bufs)) return FSDP_ERR_INVALID_ARG;
    if (mul_overflows(padded_numel, 4)) return FSDP_ERR_INVALID_ARG;
    const int64_t S = padded_numel / world;
    const int64_t begin = static_cast<int64_t>(rank_begin) * S, end = static_cast<int64_t>(rank_end) * S;
    if (begin == end) {
        empty = true;
        return FSDP_OK;
    }
    if (!master || !exp_avg || !exp_avg_sq || (!shard_out && n_dst == 0)) return FSDP_ERR_INVALID_ARG;
    const size_t gs = static_cast<size_t>(dtype_size(grad_dtype)), os = static_cast<size_t>(dtype_size(out_dtype));
    const size_t state_bytes = static_cast<size_t>(padded_numel) * 4;
    const size_t out_bytes = static_cast<size_t>(padded_numel) * os;
    if (!aligned(master, 4) || !aligned(exp_avg, 4) || !aligned(exp_avg_sq, 4) || !aligned(shard_out, os))
        return FSDP_ERR_ALIGNMENT;
    if (nonfinite_count && !aligned(nonfinite_count, 4)) return FSDP_ERR_ALIGNMENT;
    // every written buffer: master, m, v, shard_out (if any), the gathered buffers
    const void *written[3 + 1 + FSDP_MAX_WORLD];
    size_t wbytes[3 + 1 + FSDP_MAX_WORLD];
    int nw = 0;
    written[nw] = master; wbytes[nw++] = state_bytes;
    written[nw] = exp_avg; wbytes[nw++] = state_bytes;
    written[nw] = exp_avg_sq; wbytes[nw++] = state_bytes;
    if (shard_out) { written[nw] = shard_out; wbytes[nw++] = out_bytes; }
    for (int d = 0; d < n_dst; ++d) {
        if (!full_bufs[d]) return FSDP_ERR_INVALID_ARG;
        if (!aligned(full_bufs[d], os)) return FSDP_ERR_ALIGNMENT;
        written[nw] = full_bufs[d]; wbytes[nw++] = out_bytes;
    }
    for (int i = 0; i < nw; ++i)
        for (int k = i + 1; k < nw; ++k)
            if (overlaps(written[i], wbytes[i], written[k], wbytes[k])) return FSDP_ERR_INVALID_ARG;
    memset(&a, 0, sizeof(a));
    for (int q = 0; q < world; ++q) {
        if (!grads[q]) return FSDP_ERR_INVALID_ARG;
        if (!aligned(grads[q], gs)) return FSDP_ERR_ALIGNMENT;
        for (int i = 0; i < nw; ++i)
            if (overlaps(grads[q], padded_numel * gs, written[i], wbytes[i])) return FSDP_ERR_INVALID_ARG;
        a.grads[q] = grads[q];
    }
    a.master = master;
    a.m = exp_avg;
    a.v = exp_avg_sq;
    a.out = shard_out;
    a.nonfinite = nonfinite_count;
    a.begin = begin;
    a.end = end;
    a.s = make_scalars(*hp, world);
    a.world = world;
    a.n_full = n_dst;
    for (int d = 0; d < n_dst; ++d) a.full[d] = full_bufs[d];
    return FSDP_OK;
}

fsdp_status launch_rsa(const RsaArgs &a, fsdp_dtype grad_dtype, fsdp_dtype out_dtype, cudaStream_t s) {
    switch (grad_dtype) {
        case FSDP_BF16: return launch_rsa_bf16(a, out_dtype, s);
        case FSDP_F16: return launch_rsa_f16(a, out_dtype, s);
        default: return launch_rsa_f32(a, out_dtype, s);
    }
}

fsdp_status rsa_entry(const void *const *grads, fsdp_dtype grad_dtype, int world, int64_t padded_numel,
                      float *master, float *exp_avg, float *exp_avg_sq, void *shard_out, fsdp_dtype out_dtype,
                      void *const *full_bufs, int n_dst, const fsdp_adamw_hparams *hp, int rank_begin,
                      int rank_end, uint32_t *nonfinite_count, void *stream) {
    RsaArgs a;
    bool empty = false;
    const fsdp_status st = prepare_rsa(grads, grad_dtype, world, padded_numel, master, exp_avg, exp_avg_sq,
                                       shard_out, out_dtype, full_bufs, n_dst, hp, rank_begin, rank_end,
                                       nonfinite_count, a, empty);
    if (st != FSDP_OK || empty) return st;
    return launch_rsa(a, grad_dtype, out_dtype, static_cast<cudaStream_t>(stream));
}

// Validation of an all-gather: fills its arguments or sets `empty`.
// `timeouts` (device, may be NULL) counts the call's bounded waits that gave up.
fsdp_status prepare_gather(const void *shard_out, fsdp_dtype dtype, int world, int64_t padded_numel,
                           void *const *full_bufs, int n_dst, uint32_t *timeouts, ResidencyMemo &res,
                           GatherArgs &a, bool &empty) {
    empty = false;
    if (!dtype_valid(dtype)) return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (world < 1 || padded_numel < 0 || padded_numel % world != 0) return FSDP_ERR_INVALID_ARG;
    if (n_dst < 1 || n_dst > FSDP_MAX_WORLD || !full_bufs) return FSDP_ERR_INVALID_ARG;
    if (timeouts && !aligned(timeouts, 4)) return FSDP_ERR_ALIGNMENT;
    const size_t es = static_cast<size_t>(dtype_size(dtype));
    if (mul_overflows(padded_numel, static_cast<int64_t>(es))) return FSDP_ERR_INVALID_ARG;
    if (padded_numel == 0) {
        empty = true;
        return FSDP_OK;
    }
    const size_t nbytes = static_cast<size_t>(padded_numel) * es;
    if (!shard_out) return FSDP_ERR_INVALID_ARG;
    if (!aligned(shard_out, es)) return FSDP_ERR_ALIGNMENT;
    memset(&a, 0, sizeof(a));
    a.src = shard_out;
    a.nbytes = static_cast<int64_t>(nbytes);
    a.n_dst = n_dst;
    a.timeouts = timeouts;
    for (int d = 0; d < n_dst; ++d) {
        if (!full_bufs[d]) return FSDP_ERR_INVALID_ARG;
        if (!aligned(full_bufs[d], es)) return FSDP_ERR_ALIGNMENT;
        if (overlaps(full_bufs[d], nbytes, shard_out, nbytes)) return FSDP_ERR_INVALID_ARG;
        for (int e = 0; e < d; ++e)
            if (overlaps(full_bufs[d], nbytes, full_bufs[e], nbytes)) return FSDP_ERR_INVALID_ARG;
        a.dst[d] = full_bufs[d];
    }
    // the bulk-copy pipeline moves device memory only: host buffers are refused
    if (res.host_resident(shard_out)) return FSDP_ERR_INVALID_ARG;
    for (int d = 0; d < n_dst; ++d)
        if (res.host_resident(full_bufs[d])) return FSDP_ERR_INVALID_ARG;
    return FSDP_OK;
}

// Validation of a variant step (fsdp_reduce_scatter_step and the variant
// multi-unit step): fills the kernel's arguments, or sets `empty`.
struct StepPlan {
    StepArgs args;
    fsdp_dtype grad_dtype, out_dtype, state_dtype;
    int optimizer;
    bool empty;
};

fsdp_status prepare_step(const void *const *grads, fsdp_dtype grad_dtype, int world, int64_t padded_numel,
                         void *param, void *state0, void *state1, fsdp_dtype state_dtype, void *shard_out,
                         fsdp_dtype out_dtype, const fsdp_step_config *cfg, int rank_begin, int rank_end,
                         uint32_t *nonfinite_count, StepPlan &p) {
    p.empty = false;
    if (!dtype_valid(grad_dtype) || !dtype_valid(out_dtype) || !dtype_valid(state_dtype))
        return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (world < 1 || world > FSDP_MAX_WORLD || !grads || !cfg) return FSDP_ERR_INVALID_ARG;
    if (cfg->optimizer < FSDP_OPT_ADAMW || cfg->optimizer > FSDP_OPT_ADADELTA) return FSDP_ERR_INVALID_ARG;
    if (cfg->reduce_dtype != FSDP_F32 && cfg->reduce_dtype != grad_dtype) return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (state_dtype != FSDP_F32 && out_dtype != state_dtype) return FSDP_ERR_UNSUPPORTED_DTYPE;
    if (padded_numel < 0 || padded_numel % world != 0) return FSDP_ERR_INVALID_ARG;
    if (rank_begin < 0 || rank_begin > rank_end || rank_end > world) return FSDP_ERR_INVALID_ARG;
    if (cfg->step < 1 || !(cfg->grad_scale > 0.0f) || !isfinite(cfg->grad_scale)) return FSDP_ERR_INVALID_ARG;
    if (mul_overflows(padded_numel, 4)) return FSDP_ERR_INVALID_ARG;
    const int64_t S = padded_numel / world;
    const int64_t begin = static_cast<int64_t>(rank_begin) * S, end = static_cast<int64_t>(rank_end) * S;
    if (begin == end) {
        p.empty = true;
        return FSDP_OK;
    }
    const bool sgd = cfg->optimizer == FSDP_OPT_SGD;
    if (sgd ? state1 != nullptr : state1 == nullptr) return FSDP_ERR_INVALID_ARG;
    if (state_dtype == FSDP_F32 ? shard_out == nullptr : shard_out != nullptr) return FSDP_ERR_INVALID_ARG;
    if (!param || !state0) return FSDP_ERR_INVALID_ARG;
    const size_t gs = static_cast<size_t>(dtype_size(grad_dtype)), ss = static_cast<size_t>(dtype_size(state_dtype));
    const size_t os = static_cast<size_t>(dtype_size(out_dtype));
    if (!aligned(param, ss) || !aligned(state0, ss) || !aligned(state1, ss) || !aligned(shard_out, os))
        return FSDP_ERR_ALIGNMENT;
    if (nonfinite_count && !aligned(nonfinite_count, 4)) return FSDP_ERR_ALIGNMENT;
    const void *written[4] = {param, state0, state1, shard_out};
    const size_t wbytes[4] = {padded_numel * ss, padded_numel * ss, state1 ? padded_numel * ss : 0,
                              shard_out ? padded_numel * os : 0};
    for (int i = 0; i < 4; ++i)
        for (int k = i + 1; k < 4; ++k)
            if (overlaps(written[i], wbytes[i], written[k], wbytes[k])) return FSDP_ERR_INVALID_ARG;
    StepArgs &a = p.args;
    memset(&a, 0, sizeof(a));
    for (int q = 0; q < world; ++q) {
        if (!grads[q]) return FSDP_ERR_INVALID_ARG;
        if (!aligned(grads[q], gs)) return FSDP_ERR_ALIGNMENT;
        for (int i = 0; i < 4; ++i)
            if (overlaps(grads[q], padded_numel * gs, written[i], wbytes[i])) return FSDP_ERR_INVALID_ARG;
        a.grads[q] = grads[q];
    }
    a.param = param;
    a.s0 = state0;
    a.s1 = state1;
    a.out = shard_out;
    a.nonfinite = nonfinite_count;
    a.begin = begin;
    a.end = end;
    a.k = make_step_scalars(*cfg, world);
    a.world = world;
    a.reduce_lowp = cfg->reduce_dtype != FSDP_F32 ? 1 : 0;
    p.grad_dtype = grad_dtype;
    p.out_dtype = out_dtype;
    p.state_dtype = state_dtype;
    p.optimizer = cfg->optimizer;
    return FSDP_OK;
}

fsdp_status launch_step(const StepPlan &p, cudaStream_t s) {
    switch (p.optimizer) {
        case FSDP_OPT_ADAMW: return launch_step_adamw(p.args, p.grad_dtype, p.out_dtype, p.state_dtype, s);
        case FSDP_OPT_SGD: return launch_step_sgd(p.args, p.grad_dtype, p.out_dtype, p.state_dtype, s);
        case FSDP_OPT_ADAMAX: return launch_step_adamax(p.args, p.grad_dtype, p.out_dtype, p.state_dtype, s);
        default: return launch_step_adadelta(p.args, p.grad_dtype, p.out_dtype, p.state_dtype, s);
    }
}

// One unit of fsdp_step_units, validated and ready to launch.
struct UnitPlan {
    bool variant;   // the variant step (StepPlan) rather than the fused AdamW kernel
    RsaArgs rsa;
    StepPlan step;
    GatherArgs gather;
    fsdp_dtype grad_dtype, out_dtype;
    bool empty;
    int separate_gathers;
};

struct Span {
    uintptr_t lo, hi;
    bool operator<(const Span &o) const { return lo < o.lo; }
};

// Side streams of fsdp_step_units. The units of a model are independent, so
// their launches are spread round-robin over kUnitStreams streams that fork
// from the caller's stream (an event) and join back into it (one event per
// side stream): one unit's kernels then overlap the ramp-up and tail of its
// neighbours'. Per host thread and device, created on first use and kept (a
// cache, like the SM count); per thread so that concurrent callers never
// re-record each other's fork and join events.
#ifndef FSDP_UNIT_STREAMS
#define FSDP_UNIT_STREAMS 2
#endif
constexpr int kUnitStreams = FSDP_UNIT_STREAMS;

struct SideStreams {
    cudaStream_t s[kUnitStreams > 0 ? kUnitStreams : 1] = {};
    cudaEvent_t fork = nullptr;
    cudaEvent_t done[kUnitStreams > 0 ? kUnitStreams : 1] = {};
    bool ready = false;
    ~SideStreams() {
        // at thread or process exit; errors (a context already gone) are moot
        for (int i = 0; i < kUnitStreams; ++i) {
            if (s[i]) cudaStreamDestroy(s[i]);
            if (done[i]) cudaEventDestroy(done[i]);
        }
        if (fork) cudaEventDestroy(fork);
    }
};

thread_local SideStreams t_side[kMaxDevices];

fsdp_status side_streams(SideStreams *&out) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return FSDP_ERR_INVALID_ARG;
    SideStreams &x = t_side[dev];
    if (!x.ready) {
        cudaError_t e = cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming);
        for (int i = 0; i < kUnitStreams && e == cudaSuccess; ++i) {
            e = cudaStreamCreateWithFlags(&x.s[i], cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&x.done[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_status(e);
        x.ready = true;
    }
    out = &x;
    return FSDP_OK;
}

// Under stream capture: the graph node of the kernel just launched on s, the
// one node the capture's dependency set holds right after that launch.
fsdp_status last_captured_node(cudaStream_t s, cudaGraphNode_t *node) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t *deps = nullptr;
    size_t nd = 0;
    if (cudaError_t e = cudaStreamGetCaptureInfo(s, &cs, nullptr, nullptr, &deps, nullptr, &nd); e != cudaSuccess)
        return cuda_status(e);
    if (cs != cudaStreamCaptureStatusActive || nd != 1 || !deps) return FSDP_ERR_CUDA;
    *node = deps[0];
    return FSDP_OK;
}

// Launch one unit's kernels on s. Under stream capture, *update_node (if
// given) receives the graph node of the unit's update kernel.
fsdp_status launch_unit(const UnitPlan &p, cudaStream_t s, cudaGraphNode_t *update_node = nullptr) {
    fsdp_status st = p.variant ? launch_step(p.step, s) : launch_rsa(p.rsa, p.grad_dtype, p.out_dtype, s);
    if (st == FSDP_OK && update_node) st = last_captured_node(s, update_node);
    for (int k = 0; st == FSDP_OK && k < p.separate_gathers; ++k) st = launch_gather(p.gather, s);
    return st;
}

// A group of small units stepped by one batched update (the fused AdamW
// kernel's, or the variant kernel's) and `gathers` batched all-gathers
// (group.cuh), and the plan's work items: a unit's own kernels, or a
// group's.
struct Group {
    bool variant = false;
    bool fused = false;        // the fused AdamW update with the first gather fused in
    RsaGroupArgs rsa;
    RsaFusedGroupArgs fused_rsa;
    StepGroupArgs step;
    GatherGroupArgs gather;
    int n = 0;
    int64_t update_grid = 0, gather_grid = 0;
    int gathers = 0;
    int first_unit = -1;
    int optimizer = 0;
    fsdp_dtype grad_dtype = FSDP_BF16, out_dtype = FSDP_BF16, state_dtype = FSDP_F32;
};

struct Work {
    int unit = -1;            // plan index of a unit launched on its own
    Group *group = nullptr;   // or the group launched together
};

// The update node of a captured work item and what its arguments hold: the
// per-unit fused kernel (RsaArgs), the per-unit variant kernel (StepArgs),
// or the batched update of either (RsaGroupArgs, StepGroupArgs), or the
// batched fused kernel with the first gather fused in (RsaFusedGroupArgs).
enum NodeKind { kNodeUnit = 0, kNodeVariant = 1, kNodeGroup = 2, kNodeVariantGroup = 3, kNodeFusedGroup = 4 };
struct UpdateNode {
    cudaGraphNode_t node = nullptr;
    int kind = kNodeUnit;
    int world = 0;
    int grad_dtype = 0;
};

// What batched units must share: the update (fused AdamW, or the variant
// kernel with its optimizer, state dtype and reduction), N, the dtypes and
// the number of gathers (each unit keeps its own gathered buffers, 1 to
// kGroupMaxWorld of them).
struct GroupKey {
    bool variant, fused;
    int optimizer, state_dtype, reduce_lowp, world, grad_dtype, out_dtype, gathers;
    bool operator==(const GroupKey &o) const {
        return variant == o.variant && fused == o.fused && optimizer == o.optimizer && state_dtype == o.state_dtype &&
               reduce_lowp == o.reduce_lowp && world == o.world && grad_dtype == o.grad_dtype &&
               out_dtype == o.out_dtype && gathers == o.gathers;
    }
};

GroupKey key_of(const UnitPlan &p) {
    GroupKey k{};
    k.variant = p.variant;
    k.fused = !p.variant && p.rsa.n_full > 0;
    k.optimizer = p.variant ? p.step.optimizer : FSDP_OPT_ADAMW;
    k.state_dtype = p.variant ? p.step.state_dtype : FSDP_F32;
    k.reduce_lowp = p.variant ? p.step.args.reduce_lowp : 0;
    k.world = p.variant ? p.step.args.world : p.rsa.world;
    k.grad_dtype = p.grad_dtype;
    k.out_dtype = p.out_dtype;
    k.gathers = p.separate_gathers;
    return k;
}

// Whether a unit joins a batched launch: an update over all its ranks, N in
// {1, 2, 4, 8} (the builds the batched kernels are instantiated for: a
// compile-time N keeps the gradient pointers in registers), at most
// kGroupMaxNumel elements, every base pointer 16-byte
// aligned (the vector path and the bulk copies), the parameter or master in
// device memory and at most kGroupMaxWorld gathered buffers. A fused first
// gather (the fused AdamW update only) batches with the units that fuse it
// too. Larger units fill the GPU on their own and keep their own
// launches, whose gather (several tiles in flight per CTA, 3 CTAs per SM)
// measured faster at those sizes than the batched gather's one-tile CTAs.
bool groupable(const UnitPlan &p, ResidencyMemo &res) {
    if (p.empty) return false;
    const void *state = nullptr;
    if (p.variant) {
        const StepArgs &a = p.step.args;
        if (a.begin != 0 || a.end > kGroupMaxNumel) return false;
        if (a.world != 1 && a.world != 2 && a.world != 4 && a.world != 8) return false;
        if (!aligned(a.param, 16) || !aligned(a.s0, 16) || !aligned(a.s1, 16) || !aligned(a.out, 16)) return false;
        for (int q = 0; q < a.world; ++q)
            if (!aligned(a.grads[q], 16)) return false;
        state = a.param;
    } else {
        const RsaArgs &a = p.rsa;
        if (a.n_full > kGroupMaxWorld || a.begin != 0 || a.end > kGroupMaxNumel) return false;
        if (a.world != 1 && a.world != 2 && a.world != 4 && a.world != 8) return false;
        if (!aligned(a.master, 16) || !aligned(a.m, 16) || !aligned(a.v, 16) || !aligned(a.out, 16)) return false;
        for (int q = 0; q < a.world; ++q)
            if (!aligned(a.grads[q], 16)) return false;
        for (int d = 0; d < a.n_full; ++d)
            if (!aligned(a.full[d], 16)) return false;
        state = a.master;
    }
    if (p.separate_gathers > 0) {
        const GatherArgs &g = p.gather;
        if (g.n_dst < 1 || g.n_dst > kGroupMaxWorld || !aligned(g.src, 16)) return false;
        for (int d = 0; d < g.n_dst; ++d)
            if (!aligned(g.dst[d], 16)) return false;
    }
    return !res.host_resident(state);
}

Group *new_group(std::vector<std::unique_ptr<Group>> &groups, const UnitPlan &p, int u) {
    groups.push_back(std::unique_ptr<Group>(new Group()));
    Group *g = groups.back().get();
    memset(&g->rsa, 0, sizeof(g->rsa));
    memset(&g->fused_rsa, 0, sizeof(g->fused_rsa));
    memset(&g->step, 0, sizeof(g->step));
    memset(&g->gather, 0, sizeof(g->gather));
    g->variant = p.variant;
    if (p.variant) {  // every unit of a group has the same hyperparameters, N and reduction
        g->step.k = p.step.args.k;
        g->step.reduce_lowp = p.step.args.reduce_lowp;
        g->step.world = p.step.args.world;
        g->step.nonfinite = p.step.args.nonfinite;
        g->optimizer = p.step.optimizer;
        g->state_dtype = p.step.state_dtype;
    } else if (p.rsa.n_full > 0) {
        g->fused = true;
        g->fused_rsa.s = p.rsa.s;
        g->fused_rsa.world = p.rsa.world;
        g->fused_rsa.nonfinite = p.rsa.nonfinite;
    } else {
        g->rsa.s = p.rsa.s;
        g->rsa.world = p.rsa.world;
        g->rsa.nonfinite = p.rsa.nonfinite;
    }
    g->gathers = p.separate_gathers;
    g->gather.timeouts = p.gather.timeouts;  // the call's counter: the same for every unit
    g->first_unit = u;
    g->grad_dtype = p.grad_dtype;
    g->out_dtype = p.out_dtype;
    return g;
}

void add_to_group(Group &G, const UnitPlan &p) {
    const int k = G.n;
    if (G.variant) {
        const StepArgs &a = p.step.args;
        StepGroupUnit &gu = G.step.u[k];
        memset(&gu, 0, sizeof(gu));
        for (int q = 0; q < a.world; ++q) gu.grads[q] = a.grads[q];
        gu.param = a.param;
        gu.s0 = a.s0;
        gu.s1 = a.s1;
        gu.out = a.out;
        gu.numel = a.end;
        gu.cta_begin = G.update_grid;
        gu.ncta = group_update_ctas(a.end);
        G.update_grid += gu.ncta;
        G.step.n = k + 1;
    } else if (G.fused) {
        const RsaArgs &a = p.rsa;
        FusedGroupUnit &gu = G.fused_rsa.u[k];
        memset(&gu, 0, sizeof(gu));
        for (int q = 0; q < a.world; ++q) gu.grads[q] = a.grads[q];
        for (int d = 0; d < a.n_full; ++d) gu.full[d] = a.full[d];
        gu.master = a.master;
        gu.m = a.m;
        gu.v = a.v;
        gu.out = a.out;
        gu.numel = a.end;
        gu.cta_begin = G.update_grid;
        gu.ncta = group_update_ctas(a.end);
        gu.n_full = a.n_full;
        G.update_grid += gu.ncta;
        G.fused_rsa.n = k + 1;
    } else {
        const RsaArgs &a = p.rsa;
        GroupUnit &gu = G.rsa.u[k];
        memset(&gu, 0, sizeof(gu));
        for (int q = 0; q < a.world; ++q) gu.grads[q] = a.grads[q];
        gu.master = a.master;
        gu.m = a.m;
        gu.v = a.v;
        gu.out = a.out;
        gu.numel = a.end;
        gu.cta_begin = G.update_grid;
        gu.ncta = group_update_ctas(a.end);
        G.update_grid += gu.ncta;
        G.rsa.n = k + 1;
    }
    if (G.gathers > 0) {
        GatherGroupUnit &gg = G.gather.u[k];
        memset(&gg, 0, sizeof(gg));
        gg.src = p.gather.src;
        for (int d = 0; d < p.gather.n_dst; ++d) gg.dst[d] = p.gather.dst[d];
        gg.nbytes = p.gather.nbytes;
        gg.n_dst = p.gather.n_dst;
        gg.tile_begin = G.gather_grid;
        G.gather_grid += group_gather_tiles(p.gather.nbytes);
        G.gather.n = k + 1;
    }
    G.n = k + 1;
}

// The work items of a plan, in the order of each item's first unit: units
// that qualify are batched with the earlier ones of the same key
// (kGroupMax per group), a group of one is launched as that unit alone, and
// every other unit keeps its own kernels.
void make_work(const std::vector<UnitPlan> &plan, std::vector<Work> &work,
               std::vector<std::unique_ptr<Group>> &groups, ResidencyMemo &res) {
    work.clear();
    groups.clear();
    std::vector<std::pair<GroupKey, Group *>> open;  // the group now filling, per key
    for (size_t u = 0; u < plan.size(); ++u) {
        const UnitPlan &p = plan[u];
        if (p.empty) continue;
        if (!groupable(p, res)) {
            work.push_back({static_cast<int>(u), nullptr});
            continue;
        }
        const GroupKey key = key_of(p);
        std::pair<GroupKey, Group *> *slot = nullptr;
        for (auto &o : open)
            if (o.first == key) slot = &o;
        if (!slot || slot->second->n == (slot->second->fused ? kFusedGroupMax : kGroupMax)) {
            Group *g = new_group(groups, p, static_cast<int>(u));
            work.push_back({-1, g});
            if (slot) {
                slot->second = g;
            } else {
                open.push_back({key, g});
                slot = &open.back();
            }
        }
        add_to_group(*slot->second, p);
    }
    for (Work &w : work)
        if (w.group && w.group->n == 1) {
            w.unit = w.group->first_unit;
            w.group = nullptr;
        }
}

fsdp_status launch_step_group(const Group &G, cudaStream_t s) {
    switch (G.optimizer) {
        case FSDP_OPT_ADAMW:
            return launch_step_group_adamw(G.step, G.grad_dtype, G.out_dtype, G.state_dtype, G.update_grid, s);
        case FSDP_OPT_SGD:
            return launch_step_group_sgd(G.step, G.grad_dtype, G.out_dtype, G.state_dtype, G.update_grid, s);
        case FSDP_OPT_ADAMAX:
            return launch_step_group_adamax(G.step, G.grad_dtype, G.out_dtype, G.state_dtype, G.update_grid, s);
        default:
            return launch_step_group_adadelta(G.step, G.grad_dtype, G.out_dtype, G.state_dtype, G.update_grid, s);
    }
}

// Launch one work item on s; under capture, *node receives its update node.
fsdp_status launch_work(const std::vector<UnitPlan> &plan, const Work &w, cudaStream_t s, UpdateNode *node) {
    if (!w.group) {
        const UnitPlan &p = plan[static_cast<size_t>(w.unit)];
        if (node) {
            node->kind = p.variant ? kNodeVariant : kNodeUnit;
            node->world = p.variant ? p.step.args.world : p.rsa.world;
            node->grad_dtype = p.grad_dtype;
        }
        return launch_unit(p, s, node ? &node->node : nullptr);
    }
    const Group &G = *w.group;
    fsdp_status st = G.variant ? launch_step_group(G, s)
                     : G.fused ? launch_rsa_fused_group(G.fused_rsa, G.grad_dtype, G.out_dtype, G.update_grid, s)
                               : launch_rsa_group(G.rsa, G.grad_dtype, G.out_dtype, G.update_grid, s);
    if (st == FSDP_OK && node) {
        node->kind = G.variant ? kNodeVariantGroup : G.fused ? kNodeFusedGroup : kNodeGroup;
        node->world = G.variant ? G.step.world : G.fused ? G.fused_rsa.world : G.rsa.world;
        node->grad_dtype = G.grad_dtype;
        st = last_captured_node(s, &node->node);
    }
    for (int k = 0; st == FSDP_OK && k < G.gathers; ++k) st = launch_gather_group(G.gather, G.gather_grid, s);
    return st;
}

void add_span(std::vector<Span> &spans, const void *p, uintptr_t bytes) {
    if (p && bytes) spans.push_back({reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + bytes});
}

// A model step's units after validation: one plan per unit, the byte ranges
// the units write and read, and the work items (a unit's own kernels, or a
// group of small units batched into one launch per kernel) in launch order.
struct ModelPlan {
    std::vector<UnitPlan> units;
    std::vector<Span> writes;  // parameter / master, optimizer states, shard_out, gathered buffers
    std::vector<Span> reads;   // gradients
    std::vector<Work> work;
    std::vector<std::unique_ptr<Group>> groups;
};

// Refuse a model whose units share memory that one of them writes: two
// written ranges that overlap, or a gradient range that overlaps a written
// range. Different units run at the same time (side streams, batched
// launches), so either would race. Gradients shared by several units (read
// only) are fine; a unit's gradients against its own written buffers are
// also refused by that unit's own validation.
fsdp_status check_spans(ModelPlan &m) {
    std::vector<Span> &w = m.writes;
    std::sort(w.begin(), w.end());
    for (size_t i = 1; i < w.size(); ++i)
        if (w[i].lo < w[i - 1].hi) return FSDP_ERR_INVALID_ARG;
    // the written ranges are now disjoint and sorted by start, hence by end
    // too: the first one that ends after a read range starts is the only
    // one that can overlap it
    for (const Span &r : m.reads) {
        auto it = std::upper_bound(w.begin(), w.end(), r.lo, [](uintptr_t x, const Span &y) { return x < y.hi; });
        if (it != w.end() && it->lo < r.hi) return FSDP_ERR_INVALID_ARG;
    }
    return FSDP_OK;
}

// The last step of validating a model: the overlap checks, then the work items.
fsdp_status finish_plan(ModelPlan &m, ResidencyMemo &res) {
    if (fsdp_status st = check_spans(m); st != FSDP_OK) return st;
    make_work(m.units, m.work, m.groups, res);
    return FSDP_OK;
}

// The kernel launches of a validated model.
int64_t count_launches(const ModelPlan &m) {
    int64_t n = 0;
    for (const Work &w : m.work)
        n += 1 + (w.group ? w.group->gathers : m.units[static_cast<size_t>(w.unit)].separate_gathers);
    return n;
}

// Enqueue a validated model's work items in order, spread over the side
// streams when there are two or more. Under stream capture, `nodes` (if
// given) receives each work item's update node.
fsdp_status run_units(const ModelPlan &m, cudaStream_t s, std::vector<UpdateNode> *nodes = nullptr) {
    const std::vector<Work> &work = m.work;
    if (nodes) nodes->assign(work.size(), UpdateNode());
    auto node_of = [&](size_t i) { return nodes ? &(*nodes)[i] : nullptr; };
    const int busy = static_cast<int>(work.size());
    if (kUnitStreams < 2 || busy < 2) {
        for (size_t i = 0; i < work.size(); ++i)
            if (fsdp_status st = launch_work(m.units, work[i], s, node_of(i)); st != FSDP_OK) return st;
        return FSDP_OK;
    }
    SideStreams *side = nullptr;
    if (fsdp_status st = side_streams(side); st != FSDP_OK) return st;
    const int ns = busy < kUnitStreams ? busy : kUnitStreams;
    if (cudaError_t e = cudaEventRecord(side->fork, s); e != cudaSuccess) return cuda_status(e);
    for (int i = 0; i < ns; ++i)
        if (cudaError_t e = cudaStreamWaitEvent(side->s[i], side->fork, 0); e != cudaSuccess) return cuda_status(e);
    fsdp_status result = FSDP_OK;
    for (size_t i = 0; i < work.size(); ++i) {
        result = launch_work(m.units, work[i], side->s[i % ns], node_of(i));
        if (result != FSDP_OK) break;
    }
    // join every side stream back into the caller's stream, also after a
    // failed launch, so that what was enqueued stays ordered before the
    // caller's later work
    for (int i = 0; i < ns; ++i) {
        cudaError_t e = cudaEventRecord(side->done[i], side->s[i]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, side->done[i], 0);
        if (e != cudaSuccess && result == FSDP_OK) result = cuda_status(e);
    }
    return result;
}

// Validation of fsdp_step_units' units (and of a captured or planned
// step's): a plan per unit, the written and read ranges, the work items.
fsdp_status plan_units(const fsdp_unit *units, int n_units, const fsdp_adamw_hparams *hp, int gathers,
                       int fuse_first_gather, uint32_t *nonfinite_count, uint32_t *wait_timeouts, ModelPlan &m) {
    if (n_units < 0 || (n_units > 0 && !units) || !hp) return FSDP_ERR_INVALID_ARG;
    if (gathers < 0 || gathers > FSDP_MAX_WORLD) return FSDP_ERR_INVALID_ARG;
    if (wait_timeouts && !aligned(wait_timeouts, 4)) return FSDP_ERR_ALIGNMENT;
    const bool fuse = fuse_first_gather != 0 && gathers > 0;
    m.units.assign(static_cast<size_t>(n_units), UnitPlan());
    m.writes.clear();
    m.reads.clear();
    ResidencyMemo res;
    for (int u = 0; u < n_units; ++u) {
        const fsdp_unit &x = units[u];
        UnitPlan &p = m.units[static_cast<size_t>(u)];
        p.variant = false;
        if (!dtype_valid(x.grad_dtype) || !dtype_valid(x.out_dtype)) return FSDP_ERR_UNSUPPORTED_DTYPE;
        p.grad_dtype = static_cast<fsdp_dtype>(x.grad_dtype);
        p.out_dtype = static_cast<fsdp_dtype>(x.out_dtype);
        if (x.n_full < 0 || x.n_full > FSDP_MAX_WORLD || (x.n_full > 0 && !x.full_bufs)) return FSDP_ERR_INVALID_ARG;
        if (gathers > 0 && x.n_full < 1) return FSDP_ERR_INVALID_ARG;
        if (x.padded_numel > 0 && !x.shard_out) return FSDP_ERR_INVALID_ARG;
        fsdp_status st = prepare_rsa(x.grads, p.grad_dtype, x.world, x.padded_numel, x.master, x.exp_avg,
                                     x.exp_avg_sq, x.shard_out, p.out_dtype, fuse ? x.full_bufs : nullptr,
                                     fuse ? x.n_full : 0, hp, 0, x.world, nonfinite_count, p.rsa, p.empty);
        if (st != FSDP_OK) return st;
        p.separate_gathers = p.empty ? 0 : gathers - (fuse ? 1 : 0);
        if (p.separate_gathers > 0) {
            bool gempty = false;
            st = prepare_gather(x.shard_out, p.out_dtype, x.world, x.padded_numel, x.full_bufs, x.n_full,
                                wait_timeouts, res, p.gather, gempty);
            if (st != FSDP_OK) return st;
        }
        if (p.empty) continue;
        const uintptr_t P = static_cast<uintptr_t>(x.padded_numel);
        const uintptr_t sb = P * 4;
        const uintptr_t ob = P * static_cast<uintptr_t>(dtype_size(p.out_dtype));
        const uintptr_t gb = P * static_cast<uintptr_t>(dtype_size(p.grad_dtype));
        add_span(m.writes, x.master, sb);
        add_span(m.writes, x.exp_avg, sb);
        add_span(m.writes, x.exp_avg_sq, sb);
        add_span(m.writes, x.shard_out, ob);
        if (gathers > 0)
            for (int d = 0; d < x.n_full; ++d) add_span(m.writes, x.full_bufs[d], ob);
        for (int q = 0; q < x.world; ++q) add_span(m.reads, x.grads[q], gb);
    }
    return finish_plan(m, res);
}

// Validation of fsdp_step_units_ex's units (and of a captured or planned
// variant step's).
fsdp_status plan_units_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg, int gathers,
                          uint32_t *nonfinite_count, uint32_t *wait_timeouts, ModelPlan &m) {
    if (n_units < 0 || (n_units > 0 && !units) || !cfg) return FSDP_ERR_INVALID_ARG;
    if (gathers < 0 || gathers > FSDP_MAX_WORLD) return FSDP_ERR_INVALID_ARG;
    if (wait_timeouts && !aligned(wait_timeouts, 4)) return FSDP_ERR_ALIGNMENT;
    m.units.assign(static_cast<size_t>(n_units), UnitPlan());
    m.writes.clear();
    m.reads.clear();
    ResidencyMemo res;
    for (int u = 0; u < n_units; ++u) {
        const fsdp_unit_ex &x = units[u];
        UnitPlan &p = m.units[static_cast<size_t>(u)];
        p.variant = true;
        if (x.reserved != 0) return FSDP_ERR_INVALID_ARG;
        if (!dtype_valid(x.grad_dtype) || !dtype_valid(x.out_dtype) || !dtype_valid(x.state_dtype))
            return FSDP_ERR_UNSUPPORTED_DTYPE;
        const fsdp_dtype gd = static_cast<fsdp_dtype>(x.grad_dtype), od = static_cast<fsdp_dtype>(x.out_dtype);
        const fsdp_dtype sd = static_cast<fsdp_dtype>(x.state_dtype);
        p.grad_dtype = gd;
        p.out_dtype = od;
        if (x.n_full < 0 || x.n_full > FSDP_MAX_WORLD || (x.n_full > 0 && !x.full_bufs)) return FSDP_ERR_INVALID_ARG;
        if (gathers > 0 && x.n_full < 1) return FSDP_ERR_INVALID_ARG;
        fsdp_status st = prepare_step(x.grads, gd, x.world, x.padded_numel, x.param, x.state0, x.state1, sd,
                                      x.shard_out, od, cfg, 0, x.world, nonfinite_count, p.step);
        if (st != FSDP_OK) return st;
        p.empty = p.step.empty;
        p.separate_gathers = p.empty ? 0 : gathers;
        // the gathered shards: shard_out, or the parameter itself when the
        // state is bf16/fp16 (then it is the compute-dtype shard)
        const void *shard = sd == FSDP_F32 ? x.shard_out : x.param;
        if (p.separate_gathers > 0) {
            bool gempty = false;
            st = prepare_gather(shard, od, x.world, x.padded_numel, x.full_bufs, x.n_full, wait_timeouts, res,
                                p.gather, gempty);
            if (st != FSDP_OK) return st;
        }
        if (p.empty) continue;
        const uintptr_t P = static_cast<uintptr_t>(x.padded_numel);
        const uintptr_t sb = P * static_cast<uintptr_t>(dtype_size(sd));
        const uintptr_t ob = P * static_cast<uintptr_t>(dtype_size(od));
        const uintptr_t gb = P * static_cast<uintptr_t>(dtype_size(gd));
        add_span(m.writes, x.param, sb);
        add_span(m.writes, x.state0, sb);
        add_span(m.writes, x.state1, sb);
        add_span(m.writes, x.shard_out, ob);
        if (gathers > 0)
            for (int d = 0; d < x.n_full; ++d) add_span(m.writes, x.full_bufs[d], ob);
        for (int q = 0; q < x.world; ++q) add_span(m.reads, x.grads[q], gb);
    }
    return finish_plan(m, res);
}

// One step's scalars written into a validated model's update arguments, per
// unit and per batched group for its world size: the fused AdamW update's,
void set_adam_scalars(ModelPlan &m, const fsdp_adamw_hparams &hp) {
    for (UnitPlan &p : m.units)
        if (!p.empty) p.rsa.s = make_scalars(hp, p.rsa.world);
    for (auto &g : m.groups) {
        if (g->fused) {
            g->fused_rsa.s = make_scalars(hp, g->fused_rsa.world);
        } else {
            g->rsa.s = make_scalars(hp, g->rsa.world);
        }
    }
}

// and the variant update's (its scalars and the reduction flag).
void set_step_scalars(ModelPlan &m, const fsdp_step_config &c) {
    const int lowp = c.reduce_dtype != FSDP_F32 ? 1 : 0;
    for (UnitPlan &p : m.units) {
        if (p.empty) continue;
        p.step.args.k = make_step_scalars(c, p.step.args.world);
        p.step.args.reduce_lowp = lowp;
    }
    for (auto &g : m.groups) {
        g->step.k = make_step_scalars(c, g->step.world);
        g->step.reduce_lowp = lowp;
    }
}

// The per-step arguments of a planned or captured step, checked as the
// single-unit entry points check them.
bool adam_step_valid(const fsdp_adamw_hparams &hp) {
    return hp.step >= 1 && hp.grad_scale > 0.0f && isfinite(hp.grad_scale);
}

fsdp_status step_config_valid(const fsdp_step_config &c, int optimizer, const std::vector<int> &grad_dtypes) {
    if (c.optimizer != optimizer) return FSDP_ERR_INVALID_ARG;
    if (c.step < 1 || !(c.grad_scale > 0.0f) || !isfinite(c.grad_scale)) return FSDP_ERR_INVALID_ARG;
    for (int gd : grad_dtypes)
        if (c.reduce_dtype != FSDP_F32 && c.reduce_dtype != gd) return FSDP_ERR_UNSUPPORTED_DTYPE;
    return FSDP_OK;
}

// Capture the launches of a validated model into an instantiated graph,
// recording each work item's update node.
fsdp_status capture_units(const ModelPlan &m, cudaGraph_t &graph, cudaGraphExec_t &exec,
                          std::vector<UpdateNode> &nodes) {
    graph = nullptr;
    exec = nullptr;
    // sized before the capture begins, so that nothing allocates while it is open
    nodes.assign(m.work.size(), UpdateNode());
    cudaStream_t cs = nullptr;
    if (cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking); e != cudaSuccess) return cuda_status(e);
    // relaxed: the first launch of a kernel build queries its occupancy and
    // may set its shared-memory limit, which a stricter mode would refuse
    if (cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed); e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return cuda_status(e);
    }
    fsdp_status st = run_units(m, cs, &nodes);
    const cudaError_t ec = cudaStreamEndCapture(cs, &graph);  // always end the capture
    cudaStreamDestroy(cs);
    if (st != FSDP_OK || ec != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        graph = nullptr;
        return st != FSDP_OK ? st : cuda_status(ec);
    }
    if (cudaError_t e = cudaGraphInstantiate(&exec, graph, 0); e != cudaSuccess) {
        cudaGraphDestroy(graph);
        graph = nullptr;
        return cuda_status(e);
    }
    return FSDP_OK;
}

// Placeholder hyperparameters for validating and capturing a step whose
// launches supply their own scalars.
const fsdp_adamw_hparams kPlaceholderHp = {0.0f, 0.9f, 0.999f, 1e-8f, 0.0f, 1, 1.0f};

// Gradient dtypes of a model's non-empty units (a launch's reduction dtype
// must be fp32 or every one of them).
std::vector<int> grad_dtypes_of(const ModelPlan &m) {
    std::vector<int> d;
    for (const UnitPlan &p : m.units)
        if (!p.empty) d.push_back(p.grad_dtype);
    return d;
}

}  // namespace

extern "C" {

FSDP_API fsdp_status fsdp_reduce_scatter_adam_cast(const void *const *grads, fsdp_dtype grad_dtype, int world,
                                          int64_t padded_numel, float *master, float *exp_avg,
                                          float *exp_avg_sq, void *shard_out, fsdp_dtype out_dtype,
                                          const fsdp_adamw_hparams *hp, int rank_begin, int rank_end,
                                          uint32_t *nonfinite_count, void *stream) {
    if (!shard_out && padded_numel > 0 && rank_begin < rank_end) return FSDP_ERR_INVALID_ARG;
    return rsa_entry(grads, grad_dtype, world, padded_numel, master, exp_avg, exp_avg_sq, shard_out, out_dtype,
                     nullptr, 0, hp, rank_begin, rank_end, nonfinite_count, stream);
}

FSDP_API fsdp_status fsdp_reduce_scatter_adam_cast_gather(const void *const *grads, fsdp_dtype grad_dtype, int world,
                                                 int64_t padded_numel, float *master, float *exp_avg,
                                                 float *exp_avg_sq, void *shard_out, fsdp_dtype out_dtype,
                                                 void *const *full_bufs, int n_dst,
                                                 const fsdp_adamw_hparams *hp, int rank_begin, int rank_end,
                                                 uint32_t *nonfinite_count, void *stream) {
    if (n_dst < 1) return FSDP_ERR_INVALID_ARG;
    return rsa_entry(grads, grad_dtype, world, padded_numel, master, exp_avg, exp_avg_sq, shard_out, out_dtype,
                     full_bufs, n_dst, hp, rank_begin, rank_end, nonfinite_count, stream);
}

FSDP_API fsdp_status fsdp_reduce_scatter_step(const void *const *grads, fsdp_dtype grad_dtype, int world,
                                     int64_t padded_numel, void *param, void *state0, void *state1,
                                     fsdp_dtype state_dtype, void *shard_out, fsdp_dtype out_dtype,
                                     const fsdp_step_config *cfg, int rank_begin, int rank_end,
                                     uint32_t *nonfinite_count, void *stream) {
    StepPlan p;
    const fsdp_status st = prepare_step(grads, grad_dtype, world, padded_numel, param, state0, state1, state_dtype,
                                        shard_out, out_dtype, cfg, rank_begin, rank_end, nonfinite_count, p);
    if (st != FSDP_OK || p.empty) return st;
    return launch_step(p, static_cast<cudaStream_t>(stream));
}

FSDP_API fsdp_status fsdp_all_gather(const void *shard_out, fsdp_dtype dtype, int world, int64_t padded_numel,
                            void *const *full_bufs, int n_dst, uint32_t *wait_timeouts, void *stream) {
    GatherArgs a;
    bool empty = false;
    ResidencyMemo res;
    const fsdp_status st =
        prepare_gather(shard_out, dtype, world, padded_numel, full_bufs, n_dst, wait_timeouts, res, a, empty);
    if (st != FSDP_OK || empty) return st;
    return launch_gather(a, static_cast<cudaStream_t>(stream));
}

FSDP_API fsdp_status fsdp_step_units(const fsdp_unit *units, int n_units, const fsdp_adamw_hparams *hp,
                                     int gathers, int fuse_first_gather, uint32_t *nonfinite_count,
                                     uint32_t *wait_timeouts, void *stream) {
    return guarded([&]() -> fsdp_status {
        ModelPlan m;
        const fsdp_status st =
            plan_units(units, n_units, hp, gathers, fuse_first_gather, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return run_units(m, static_cast<cudaStream_t>(stream));
    });
}

FSDP_API fsdp_status fsdp_step_units_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                        int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                        void *stream) {
    return guarded([&]() -> fsdp_status {
        ModelPlan m;
        const fsdp_status st = plan_units_ex(units, n_units, cfg, gathers, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return run_units(m, static_cast<cudaStream_t>(stream));
    });
}

FSDP_API fsdp_status fsdp_step_units_launches(const fsdp_unit *units, int n_units, const fsdp_adamw_hparams *hp,
                                              int gathers, int fuse_first_gather, int64_t *launches_out) {
    return guarded([&]() -> fsdp_status {
        if (!launches_out) return FSDP_ERR_INVALID_ARG;
        ModelPlan m;
        const fsdp_status st = plan_units(units, n_units, hp, gathers, fuse_first_gather, nullptr, nullptr, m);
        if (st != FSDP_OK) return st;
        *launches_out = count_launches(m);
        return FSDP_OK;
    });
}

FSDP_API fsdp_status fsdp_step_units_ex_launches(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                                 int gathers, int64_t *launches_out) {
    return guarded([&]() -> fsdp_status {
        if (!launches_out) return FSDP_ERR_INVALID_ARG;
        ModelPlan m;
        const fsdp_status st = plan_units_ex(units, n_units, cfg, gathers, nullptr, nullptr, m);
        if (st != FSDP_OK) return st;
        *launches_out = count_launches(m);
        return FSDP_OK;
    });
}

}  // extern "C"

// A validated model step (fsdp_step_plan_*): the model's plan, whose update
// arguments each launch rewrites with its step's scalars. `variant` plans
// hold the variant update of one optimizer. `device` is the device that was
// current when the plan was made: its buffers' addresses belong to it.
struct fsdp_step_plan {
    ModelPlan m;
    bool variant = false;
    int optimizer = 0;
    std::vector<int> grad_dtypes;
    int device = -1;
};

// A captured model step (fsdp_step_graph_*): the instantiated graph and,
// per work item (a unit, or a group of small units in one batched launch),
// its update node with the kind of arguments it holds, its world size and
// gradient dtype, which the per-step arguments depend on. `variant` graphs
// hold the variant kernel of one optimizer.
struct fsdp_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    std::vector<UpdateNode> nodes;
    bool variant = false;
    int optimizer = 0;
};

namespace {

fsdp_status make_graph(const ModelPlan &m, bool variant, int optimizer, fsdp_step_graph **graph_out) {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    std::vector<UpdateNode> nodes;
    if (fsdp_status st = capture_units(m, graph, exec, nodes); st != FSDP_OK) return st;
    fsdp_step_graph *g = new (std::nothrow) fsdp_step_graph;
    if (!g) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return FSDP_ERR_HOST_MEMORY;
    }
    g->graph = graph;
    g->exec = exec;
    g->nodes = std::move(nodes);
    g->variant = variant;
    g->optimizer = optimizer;
    *graph_out = g;
    return FSDP_OK;
}

fsdp_status make_plan(ModelPlan &m, bool variant, int optimizer, fsdp_step_plan **plan_out) {
    fsdp_step_plan *p = new (std::nothrow) fsdp_step_plan;
    if (!p) return FSDP_ERR_HOST_MEMORY;
    p->m = std::move(m);
    p->variant = variant;
    p->optimizer = optimizer;
    p->grad_dtypes = grad_dtypes_of(p->m);
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        (void)cudaGetLastError();
        p->device = -1;
    }
    *plan_out = p;
    return FSDP_OK;
}

// Write a step's arguments into one captured update node: the node's own
// arguments (kernel params: the args struct first; for the per-unit kernels
// then int64 vbegin, nchunks, vend; the batched update has no other) with
// only the step-dependent fields replaced.
template <class Args, int NPARAMS, class Fill>
fsdp_status set_update_node(fsdp_step_graph *graph, cudaGraphNode_t node, Fill fill) {
    cudaKernelNodeParams kp;
    if (cudaError_t e = cudaGraphKernelNodeGetParams(node, &kp); e != cudaSuccess) return cuda_status(e);
    if (!kp.kernelParams) return FSDP_ERR_INVALID_ARG;
    std::unique_ptr<Args> a(new (std::nothrow) Args);  // up to ~31 KB: not on the caller's stack
    if (!a) return FSDP_ERR_HOST_MEMORY;
    memcpy(a.get(), kp.kernelParams[0], sizeof(Args));
    fill(*a);
    void *args[NPARAMS];
    args[0] = a.get();
    for (int i = 1; i < NPARAMS; ++i) args[i] = kp.kernelParams[i];
    kp.kernelParams = args;
    return cuda_status(cudaGraphExecKernelNodeSetParams(graph->exec, node, &kp));
}

}  // namespace

extern "C" {

FSDP_API fsdp_status fsdp_step_graph_create(const fsdp_unit *units, int n_units, int gathers, int fuse_first_gather,
                                            uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                            fsdp_step_graph **graph_out) {
    return guarded([&]() -> fsdp_status {
        if (!graph_out) return FSDP_ERR_INVALID_ARG;
        *graph_out = nullptr;
        // every launch writes the step's own scalars into the update nodes
        ModelPlan m;
        fsdp_status st =
            plan_units(units, n_units, &kPlaceholderHp, gathers, fuse_first_gather, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return make_graph(m, false, FSDP_OPT_ADAMW, graph_out);
    });
}

FSDP_API fsdp_status fsdp_step_graph_create_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                               int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                               fsdp_step_graph **graph_out) {
    return guarded([&]() -> fsdp_status {
        if (!graph_out) return FSDP_ERR_INVALID_ARG;
        *graph_out = nullptr;
        ModelPlan m;
        fsdp_status st = plan_units_ex(units, n_units, cfg, gathers, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return make_graph(m, true, cfg->optimizer, graph_out);
    });
}

FSDP_API fsdp_status fsdp_step_graph_launch(fsdp_step_graph *graph, const fsdp_adamw_hparams *hp, void *stream) {
    return guarded([&]() -> fsdp_status {
        if (!graph || !hp || graph->variant) return FSDP_ERR_INVALID_ARG;
        if (!adam_step_valid(*hp)) return FSDP_ERR_INVALID_ARG;
        for (const UpdateNode &n : graph->nodes) {
            const AdamScalars sc = make_scalars(*hp, n.world);
            fsdp_status st =
                n.kind == kNodeGroup ? set_update_node<RsaGroupArgs, 1>(graph, n.node, [&](RsaGroupArgs &a) { a.s = sc; })
                : n.kind == kNodeFusedGroup
                    ? set_update_node<RsaFusedGroupArgs, 1>(graph, n.node, [&](RsaFusedGroupArgs &a) { a.s = sc; })
                    : set_update_node<RsaArgs, 4>(graph, n.node, [&](RsaArgs &a) { a.s = sc; });
            if (st != FSDP_OK) return st;
        }
        return cuda_status(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
    });
}

FSDP_API fsdp_status fsdp_step_graph_launch_ex(fsdp_step_graph *graph, const fsdp_step_config *cfg, void *stream) {
    return guarded([&]() -> fsdp_status {
        if (!graph || !cfg || !graph->variant) return FSDP_ERR_INVALID_ARG;
        std::vector<int> gds;
        for (const UpdateNode &n : graph->nodes) gds.push_back(n.grad_dtype);
        if (fsdp_status st = step_config_valid(*cfg, graph->optimizer, gds); st != FSDP_OK) return st;
        const int lowp = cfg->reduce_dtype != FSDP_F32 ? 1 : 0;
        for (const UpdateNode &n : graph->nodes) {
            const StepScalars k = make_step_scalars(*cfg, n.world);
            fsdp_status st = n.kind == kNodeVariantGroup
                                 ? set_update_node<StepGroupArgs, 1>(graph, n.node,
                                                                     [&](StepGroupArgs &a) {
                                                                         a.k = k;
                                                                         a.reduce_lowp = lowp;
                                                                     })
                                 : set_update_node<StepArgs, 4>(graph, n.node, [&](StepArgs &a) {
                                       a.k = k;
                                       a.reduce_lowp = lowp;
                                   });
            if (st != FSDP_OK) return st;
        }
        return cuda_status(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
    });
}

FSDP_API fsdp_status fsdp_step_graph_destroy(fsdp_step_graph *graph) {
    if (!graph) return FSDP_OK;
    const cudaError_t e1 = graph->exec ? cudaGraphExecDestroy(graph->exec) : cudaSuccess;
    const cudaError_t e2 = graph->graph ? cudaGraphDestroy(graph->graph) : cudaSuccess;
    delete graph;
    return e1 != cudaSuccess ? cuda_status(e1) : cuda_status(e2);
}

FSDP_API fsdp_status fsdp_step_plan_create(const fsdp_unit *units, int n_units, int gathers, int fuse_first_gather,
                                           uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                           fsdp_step_plan **plan_out) {
    return guarded([&]() -> fsdp_status {
        if (!plan_out) return FSDP_ERR_INVALID_ARG;
        *plan_out = nullptr;
        ModelPlan m;
        fsdp_status st =
            plan_units(units, n_units, &kPlaceholderHp, gathers, fuse_first_gather, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return make_plan(m, false, FSDP_OPT_ADAMW, plan_out);
    });
}

FSDP_API fsdp_status fsdp_step_plan_create_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                              int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                              fsdp_step_plan **plan_out) {
    return guarded([&]() -> fsdp_status {
        if (!plan_out) return FSDP_ERR_INVALID_ARG;
        *plan_out = nullptr;
        ModelPlan m;
        fsdp_status st = plan_units_ex(units, n_units, cfg, gathers, nonfinite_count, wait_timeouts, m);
        if (st != FSDP_OK) return st;
        return make_plan(m, true, cfg->optimizer, plan_out);
    });
}

// Whether the device current now is the one a plan was made on.
static bool on_plan_device(const fsdp_step_plan *plan) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        dev = -1;
    }
    return dev == plan->device;
}

FSDP_API fsdp_status fsdp_step_plan_launch(fsdp_step_plan *plan, const fsdp_adamw_hparams *hp, void *stream) {
    if (!plan || !hp || plan->variant) return FSDP_ERR_INVALID_ARG;
    if (!adam_step_valid(*hp)) return FSDP_ERR_INVALID_ARG;
    if (!on_plan_device(plan)) return FSDP_ERR_INVALID_ARG;
    set_adam_scalars(plan->m, *hp);
    return run_units(plan->m, static_cast<cudaStream_t>(stream));
}

FSDP_API fsdp_status fsdp_step_plan_launch_ex(fsdp_step_plan *plan, const fsdp_step_config *cfg, void *stream) {
    if (!plan || !cfg || !plan->variant) return FSDP_ERR_INVALID_ARG;
    if (fsdp_status st = step_config_valid(*cfg, plan->optimizer, plan->grad_dtypes); st != FSDP_OK) return st;
    if (!on_plan_device(plan)) return FSDP_ERR_INVALID_ARG;
    set_step_scalars(plan->m, *cfg);
    return run_units(plan->m, static_cast<cudaStream_t>(stream));
}

FSDP_API fsdp_status fsdp_step_plan_destroy(fsdp_step_plan *plan) {
    delete plan;
    return FSDP_OK;
}

FSDP_API const char *fsdp_status_string(fsdp_status status) {
    switch (status) {
        case FSDP_OK: return "FSDP_OK";
        case FSDP_ERR_INVALID_ARG: return "FSDP_ERR_INVALID_ARG: invalid argument";
        case FSDP_ERR_ALIGNMENT: return "FSDP_ERR_ALIGNMENT: pointer not aligned to its element size";
        case FSDP_ERR_CUDA: return "FSDP_ERR_CUDA: a CUDA call or kernel launch failed";
        case FSDP_ERR_UNSUPPORTED_DTYPE: return "FSDP_ERR_UNSUPPORTED_DTYPE: unsupported dtype";
        case FSDP_ERR_HOST_MEMORY: return "FSDP_ERR_HOST_MEMORY: host memory for the call's bookkeeping ran out";
        default: return "FSDP_ERR_UNKNOWN: unknown status";
    }
}

FSDP_API int fsdp_last_cuda_error(void) { return g_last_cuda_error; }

FSDP_API fsdp_status fsdp_take_wait_timeouts(uint32_t *count_out) {
    if (!count_out) return FSDP_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e);
    *count_out = take_gather_wait_timeouts();
    return FSDP_OK;
}

FSDP_API fsdp_status fsdp_check_bounded_wait(int64_t limit_cycles, uint32_t *wait_timeouts, void *stream) {
    if (limit_cycles < 1 || limit_cycles > (int64_t{1} << 31)) return FSDP_ERR_INVALID_ARG;
    if (wait_timeouts && !aligned(wait_timeouts, 4)) return FSDP_ERR_ALIGNMENT;
    return launch_stalled_wait(static_cast<long long>(limit_cycles), wait_timeouts,
                               static_cast<cudaStream_t>(stream));
}

}  // extern "C"
