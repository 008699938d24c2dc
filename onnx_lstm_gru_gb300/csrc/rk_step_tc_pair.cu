// rk_step_tc_pair.cu -- the tensor-core step kernel (rk_step_tc.cuh) of Half
// layers for teams of at most 64 batch rows: two 64-wide k blocks share each
// 128-row tile, and every gate thread takes 4 units.
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_pairs(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16,
                          const CUtensorMap* ta, const CUtensorMap* tb) {
  return step_tc_mode_dispatch<1, __half>(p, plan, s, resident, h16, ta, tb);
}

}  // namespace rk
