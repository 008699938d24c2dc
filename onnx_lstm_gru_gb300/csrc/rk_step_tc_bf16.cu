// rk_step_tc_bf16.cu -- the tensor-core step kernel (rk_step_tc.cuh) of
// bfloat16 layers for teams of more than 64 batch rows (one k block per
// tile).  The kernels are the Half ones with the other element type: the
// tensor cores read bfloat16 operands (kind::f16 with the bfloat16 type
// fields) and the exchanged h is rounded to bfloat16.
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_rows(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                         __nv_bfloat16* h16, const CUtensorMap* ta, const CUtensorMap* tb) {
  return step_tc_mode_dispatch<0, __nv_bfloat16>(p, plan, s, resident, h16, ta, tb);
}

}  // namespace rk
