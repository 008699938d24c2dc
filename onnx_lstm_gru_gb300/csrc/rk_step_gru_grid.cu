// Step-kernel instantiations: GRU cell, grid exchange.
#include "rk_step_launch.cuh"

namespace rk {
template cudaError_t step_entry<1, true>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
