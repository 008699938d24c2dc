// rk_step_tc_pair_bf16.cu -- the tensor-core step kernel (rk_step_tc.cuh) of
// bfloat16 layers for teams of at most 64 batch rows (paired k blocks, flags).
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_pairs(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                          __nv_bfloat16* h16, const CUtensorMap* ta, const CUtensorMap* tb) {
  return step_tc_mode_dispatch<1, __nv_bfloat16>(p, plan, s, resident, h16, ta, tb);
}

}  // namespace rk
