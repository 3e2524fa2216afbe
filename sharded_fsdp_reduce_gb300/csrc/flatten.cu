// flatten.cu -- flatten + pad of one FSDP unit's parameters.
//
// The unit's tensors are copied back to back into one flat buffer and the
// padding at the end is zero-filled ("Fully Sharded Data Parallel: faster AI
// training with fewer GPUs", "Harnessing FSDP's full power", item 3: a wrapped
// module's parameters are flattened into a single tensor). One launch handles
// up to FlattenArgs::kBatch segments, one per blockIdx.y; a segment with a
// NULL source is zero-filled. Runs once per unit at set-up.
#include "host.cuh"

namespace fsdp {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) flatten_kernel(const __grid_constant__ FlattenArgs a) {
    const int t = blockIdx.y;
    const char *src = static_cast<const char *>(a.src[t]);
    char *dst = static_cast<char *>(a.dst) + a.dst_byte_off[t];
    const int64_t n = a.nbytes[t];
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    const int64_t nvec = vec ? n / 16 : 0;
    for (int64_t k = tid; k < nvec; k += stride) {
        const uint4 x = src ? *reinterpret_cast<const uint4 *>(src + 16 * k) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(dst + 16 * k) = x;
    }
    // the rest in 2-byte units (every element size is a multiple of 2)
    const int64_t base = 16 * nvec;
    const int64_t units = (n - base) / 2;
    for (int64_t u = tid; u < units; u += stride) {
        const uint16_t x = src ? *reinterpret_cast<const uint16_t *>(src + base + 2 * u) : uint16_t(0);
        *reinterpret_cast<uint16_t *>(dst + base + 2 * u) = x;
    }
}

}  // namespace

fsdp_status launch_flatten(const FlattenArgs &a, cudaStream_t stream) {
    if (a.count <= 0) return FSDP_OK;
    int64_t longest = 0;
    for (int t = 0; t < a.count; ++t) longest = a.nbytes[t] > longest ? a.nbytes[t] : longest;
    if (longest == 0) return FSDP_OK;
    const int64_t need = (longest / 16 + 1 + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 4;
    const unsigned gx = static_cast<unsigned>(need < cap ? need : cap);
    flatten_kernel<<<dim3(gx, a.count), kThreads, 0, stream>>>(a);
    return check_launch();
}

}  // namespace fsdp
