// Step-kernel instantiations: RNN cell, cluster exchange.
#include "rk_step_launch.cuh"

namespace rk {
template cudaError_t step_entry<2, false>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
