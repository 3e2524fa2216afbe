// rsa_bf16.cu -- instantiations of the fused reduce-scatter + AdamW + cast
// kernel for bf16 gradients (all output dtypes, N in {2, 4, 8} and generic N).
#include "rsa_launch.cuh"

namespace fsdp {
fsdp_status launch_rsa_bf16(const RsaArgs &a, int out_dtype, cudaStream_t stream) {
    return rsa::launch_grad<FSDP_BF16>(a, out_dtype, stream);
}
}  // namespace fsdp
