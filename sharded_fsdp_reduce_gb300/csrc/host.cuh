// host.cuh -- host-side plumbing of libfsdpreduce.so (not part of the ABI):
// launch sizing, per-device caches, argument checks and the internal launcher
// entry points of the kernels' translation units.
#pragma once

#include <atomic>
#include <map>

#include "common.cuh"

namespace fsdp {

// SM count of the current device, cached per device.
int sm_count();

// Ordinal of the current device (0 if it cannot be read).
inline int current_device() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 ? dev : 0;
}

// One-time per-device settings of a kernel (its shared-memory opt-in): a
// flag per device ordinal.
struct PerDeviceOnce {
    static constexpr int kMaxDevices = 64;
    std::atomic<bool> done[kMaxDevices] = {};
    bool is_done(int dev) const { return dev < kMaxDevices ? done[dev].load(std::memory_order_acquire) : false; }
    void mark(int dev) {
        if (dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
    }
};

// Record the CUDA error behind an FSDP_ERR_CUDA for fsdp_last_cuda_error().
fsdp_status cuda_status(cudaError_t e);

// Grid of a non-persistent elementwise launch: enough blocks for about
// `per_thread` work items per thread, but never less than one resident wave
// (`wave` blocks) unless there is less work than that, and at least 1.
inline int grid_for(int64_t items, int threads, int per_thread, int64_t wave) {
    const int64_t need = (items + threads - 1) / threads;  // one item per thread
    const int64_t want = (items + int64_t(threads) * per_thread - 1) / (int64_t(threads) * per_thread);
    int64_t g = want > wave ? want : (need < wave ? need : wave);
    if (g < 1) g = 1;
    if (g > 0x7fffffff) g = 0x7fffffff;
    return static_cast<int>(g);
}

// Check the launch that was just enqueued.
inline fsdp_status check_launch() { return cuda_status(cudaGetLastError()); }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Whether p is host memory (page-locked and mapped, or another host address
// the device reaches): buffers there stream over the host link, which picks
// the kernels' low-occupancy build. A pointer the runtime cannot classify
// counts as device memory (its error is cleared).
inline bool host_resident(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

// host_resident() for the many buffers of one call, with one runtime query
// per device allocation rather than per pointer: once a pointer is found in
// device memory, the driver's address range of its allocation is kept, and
// every later pointer inside that range is device memory without a query.
// Lives for one validation pass, during which the caller's allocations stay
// as they are; its answers are host_resident()'s.
class ResidencyMemo {
  public:
    bool host_resident(const void *p);

  private:
    std::map<uintptr_t, uintptr_t> device_;  // start -> end of allocations found in device memory
};

// Byte ranges [a, a+na) and [b, b+nb) overlap.
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Resident blocks per SM of a kernel, queried once per instantiation and
// cached (all devices of a process are assumed to be the same part).
template <class Kernel>
fsdp_status cached_occupancy(std::atomic<int> &cache, Kernel kernel, int threads, size_t smem, int *out) {
    int b = cache.load(std::memory_order_relaxed);
    if (b == 0) {
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem);
        if (e != cudaSuccess) return cuda_status(e);
        b = b > 0 ? b : 1;
        cache.store(b, std::memory_order_relaxed);
    }
    *out = b;
    return FSDP_OK;
}

// ---------------------------------------------------------------- internal launchers

// One translation unit per gradient dtype (rsa_bf16.cu, rsa_f16.cu, rsa_f32.cu).
// a.n_full > 0 selects the variant with the fused all-gather.
fsdp_status launch_rsa_bf16(const RsaArgs &a, int out_dtype, cudaStream_t stream);
fsdp_status launch_rsa_f16(const RsaArgs &a, int out_dtype, cudaStream_t stream);
fsdp_status launch_rsa_f32(const RsaArgs &a, int out_dtype, cudaStream_t stream);

// One translation unit per optimizer (step_adamw.cu, step_sgd.cu, ...).
fsdp_status launch_step_adamw(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s);
fsdp_status launch_step_sgd(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s);
fsdp_status launch_step_adamax(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s);
fsdp_status launch_step_adadelta(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype,
                                 cudaStream_t s);

fsdp_status launch_gather(const GatherArgs &a, cudaStream_t stream);

// Read and reset the count of bounded waits that gave up in the gather kernels.
uint32_t take_gather_wait_timeouts();
fsdp_status launch_stalled_wait(long long limit_cycles, uint32_t *per_call, cudaStream_t stream);

fsdp_status launch_flatten(const FlattenArgs &a, cudaStream_t stream);

}  // namespace fsdp
