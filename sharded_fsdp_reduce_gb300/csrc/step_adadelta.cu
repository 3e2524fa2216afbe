// step_adadelta.cu -- instantiations of the variant-step kernel for the adadelta update.
#include "step_impl.cuh"

namespace fsdp {
fsdp_status launch_step_adadelta(const StepArgs &a, int grad_dtype, int out_dtype, int state_dtype, cudaStream_t s) {
    return step::launch_opt<FSDP_OPT_ADADELTA>(a, grad_dtype, out_dtype, state_dtype, s);
}
}  // namespace fsdp
