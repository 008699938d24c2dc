// Fused step-kernel instantiations: RNN cell.
#include "rk_step_fast.cuh"

namespace rk {
template cudaError_t step_fast_entry<2>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
