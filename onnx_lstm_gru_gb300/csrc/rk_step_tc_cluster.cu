// rk_step_tc_cluster.cu -- the tensor-core step kernel (rk_step_tc.cuh) of
// Half layers for teams of at most 64 batch rows whose hidden units fit one
// thread-block cluster at 32 units per CTA: paired k-block tiles, and
// publication of h by remote mbarrier arrivals inside the cluster instead of
// global flags.
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_cluster(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16) {
  return step_tc_mode_dispatch<2, __half>(p, plan, s, resident, h16, nullptr, nullptr);
}

}  // namespace rk
