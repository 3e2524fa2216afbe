// step_group_sgd.cu -- instantiations of the batched variant-step kernel for
// the sgd update.
#include "step_group.cuh"

namespace fsdp {
fsdp_status launch_step_group_sgd(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype,
                                  int64_t grid, cudaStream_t s) {
    return step::launch_group_opt<FSDP_OPT_SGD>(g, grad_dtype, out_dtype, state_dtype, grid, s);
}
}  // namespace fsdp
