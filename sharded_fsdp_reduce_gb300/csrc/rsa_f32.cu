// rsa_f32.cu -- instantiations of the fused reduce-scatter + AdamW + cast
// kernel for f32 gradients (all output dtypes, N in {2, 4, 8} and generic N).
#include "rsa_launch.cuh"

namespace fsdp {
fsdp_status launch_rsa_f32(const RsaArgs &a, int out_dtype, cudaStream_t stream) {
    return rsa::launch_grad<FSDP_F32>(a, out_dtype, stream);
}
}  // namespace fsdp
