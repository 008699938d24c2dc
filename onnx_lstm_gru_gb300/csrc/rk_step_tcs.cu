// rk_step_tcs.cu -- the small-batch tensor-core step kernel (rk_step_tcs.cuh)
// of Half layers, its shared-memory size and the entry point.
#include "rk_step_tcs.cuh"

namespace rk {

size_t step_tcs_smem(int G, int H) { return xs_layout(G, H).total; }

cudaError_t step_tcs_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16) {
  if (p.dtype == 2) return step_tcs_bf16(p, plan, s, resident, static_cast<__nv_bfloat16*>(h16));
  return step_tcs_cells(p, plan, s, resident, static_cast<__half*>(h16));
}

}  // namespace rk
