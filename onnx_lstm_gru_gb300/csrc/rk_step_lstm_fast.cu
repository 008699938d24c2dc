// Fused step-kernel instantiations: LSTM cell.
#include "rk_step_fast.cuh"

namespace rk {
template cudaError_t step_fast_entry<0>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
