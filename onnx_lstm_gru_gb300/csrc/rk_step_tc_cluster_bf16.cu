// rk_step_tc_cluster_bf16.cu -- the tensor-core step kernel (rk_step_tc.cuh)
// of bfloat16 layers for teams of at most 64 batch rows in one thread-block
// cluster (32 units per CTA, publication by remote mbarrier arrivals).
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_cluster(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                            __nv_bfloat16* h16) {
  return step_tc_mode_dispatch<2, __nv_bfloat16>(p, plan, s, resident, h16, nullptr, nullptr);
}

}  // namespace rk
