// rk_step_tcs.cu -- the small-batch tensor-core step kernel (rk_step_tcs.cuh)
// of Half layers, its shared-memory size and the entry point.
#include "rk_step_tcs.cuh"

namespace rk {

size_t step_tcs_smem(int G, int H) { return xs_layout(G, H).total; }

cudaError_t step_tcs_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void*) {
  // the exchanged operand lives in the CTAs' shared memory, not in scratch
  if (p.dtype == 2) return step_tcs_bf16(p, plan, s, resident);
  return step_tcs_cells<__half>(p, plan, s, resident);
}

}  // namespace rk
