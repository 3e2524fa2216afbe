// step_adamax.cu -- instantiations of the variant-step kernel for the adamax update.
#include "step_impl.cuh"

namespace fsdp {
fsdp_status launch_step_adamax(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s) {
    return step::launch_opt<FSDP_OPT_ADAMAX>(a, grad_dtype, out_dtype, state_dtype, s);
}
}  // namespace fsdp
