// Fused step-kernel instantiations: GRU cell.
#include "rk_step_fast.cuh"

namespace rk {
template cudaError_t step_fast_entry<1>(const StepParams&, const StepPlan&, cudaStream_t, int*);
}  // namespace rk
