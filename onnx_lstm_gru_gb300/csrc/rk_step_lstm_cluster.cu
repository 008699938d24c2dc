// Step-kernel instantiations: LSTM cell, cluster exchange.
#include "rk_step_launch.cuh"

namespace rk {
template cudaError_t step_entry<0, false>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
