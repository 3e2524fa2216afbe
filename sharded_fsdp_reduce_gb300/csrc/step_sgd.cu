// step_sgd.cu -- instantiations of the variant-step kernel for the sgd update.
#include "step_impl.cuh"

namespace fsdp {
fsdp_status launch_step_sgd(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s) {
    return step::launch_opt<FSDP_OPT_SGD>(a, grad_dtype, out_dtype, state_dtype, s);
}
}  // namespace fsdp
