// gather.cu -- the all-gather of the compute-dtype shards.
//
// Rank r's shard is shard_out[r*S, (r+1)*S), so the concatenation of the N
// shards in rank order is shard_out itself, and every emulated rank's full
// buffer receives a copy of it ("Fully Sharded Data Parallel: faster AI
// training with fewer GPUs", "From all-reduce to sharded parameters", first
// figure caption; "FSDP (Fully Sharded Data Parallel)", "The Per-Layer
// Communication": gathered before forward and again before backward).
//
// Each thread reads one 16-byte word of the source once and writes it to the
// n_dst destinations, so the traffic is (1 + n_dst) * P_pad * sizeof(dtype)
// bytes and the kernel is HBM-write bound. A tail shorter than 16 bytes (and
// the whole copy when a pointer is not 16-byte aligned) moves in 2-byte units.
#include "common.cuh"

namespace fsdp {
namespace {

constexpr int kThreads = 256;

template <int ND>
__global__ void __launch_bounds__(kThreads)
    gather_kernel(const __grid_constant__ GatherArgs a, int64_t nvec, int64_t tail_units) {
    const int n = ND > 0 ? ND : a.n_dst;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const char *src = static_cast<const char *>(a.src);
    for (int64_t k = tid; k < nvec; k += stride) {
        const uint4 x = ld_stream(src + 16 * k);
        if constexpr (ND > 0) {
#pragma unroll
            for (int d = 0; d < ND; ++d) st_stream(static_cast<char *>(a.dst[d]) + 16 * k, x);
        } else {
            for (int d = 0; d < n; ++d) st_stream(static_cast<char *>(a.dst[d]) + 16 * k, x);
        }
    }
    // 2-byte units after the vector part
    const int64_t base = 16 * nvec;
    for (int64_t u = tid; u < tail_units; u += stride) {
        const uint16_t x = *reinterpret_cast<const uint16_t *>(src + base + 2 * u);
        for (int d = 0; d < n; ++d) *reinterpret_cast<uint16_t *>(static_cast<char *>(a.dst[d]) + base + 2 * u) = x;
    }
}

template <int ND>
fsdp_status launch_nd(const GatherArgs &a, cudaStream_t stream) {
    static int blocks_per_sm = 0;
    if (blocks_per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gather_kernel<ND>, kThreads, 0);
        if (e != cudaSuccess) return cuda_status(e);
        blocks_per_sm = b > 0 ? b : 1;
    }
    bool vec = aligned(a.src, 16);
    for (int d = 0; d < a.n_dst; ++d) vec = vec && aligned(a.dst[d], 16);
    const int64_t nvec = vec ? a.nbytes / 16 : 0;
    const int64_t tail_units = (a.nbytes - 16 * nvec) / 2;
    const int64_t items = nvec + tail_units;
    const int64_t need = (items + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
    const int grid = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
    gather_kernel<ND><<<grid, kThreads, 0, stream>>>(a, nvec, tail_units);
    return check_launch();
}

}  // namespace

fsdp_status launch_gather(const GatherArgs &a, cudaStream_t stream) {
    switch (a.n_dst) {
        case 1: return launch_nd<1>(a, stream);
        case 2: return launch_nd<2>(a, stream);
        case 4: return launch_nd<4>(a, stream);
        case 8: return launch_nd<8>(a, stream);
        default: return launch_nd<0>(a, stream);
    }
}

}  // namespace fsdp
