// rk_step_tcs_bf16.cu -- the small-batch tensor-core step kernel
// (rk_step_tcs.cuh) of bfloat16 layers.
#include "rk_step_tcs.cuh"

namespace rk {

cudaError_t step_tcs_bf16(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident) {
  return step_tcs_cells<__nv_bfloat16>(p, plan, s, resident);
}

}  // namespace rk
