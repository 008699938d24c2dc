// rk_step_tcs.cu -- the small-batch tensor-core step kernel (rk_step_tcs.cuh)
// of Half layers, its shared-memory size and the entry point.
#include "rk_step_tcs.cuh"

namespace rk {

// Dynamic shared memory of a CTA: the layout, padded so that no more CTAs
// share an SM than their TMEM allocations fit at once.  A CTA beyond that
// would wait in tcgen05.alloc for another to free its columns, and within a
// cluster the others may be waiting for it.
size_t step_tcs_smem(int G, int H, bool stacked) {
  const size_t need = xs_layout(G, H).total;
  const int per_sm = (int)(512u / tcs_tmem_cols(H, G, stacked));  // allocations that fit an SM's 512 columns
  int dev = 0, sm_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || sm_smem <= 0) {
    cudaGetLastError();
    sm_smem = 233472;  // 228 KB
  }
  const size_t floor = (size_t)sm_smem / (size_t)(per_sm + 1) + 1;
  return need > floor ? need : floor;
}

cudaError_t step_tcs_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void*) {
  // the exchanged operand lives in the CTAs' shared memory, not in scratch
  if (p.dtype == 2) return step_tcs_bf16(p, plan, s, resident);
  return step_tcs_cells<__half>(p, plan, s, resident);
}

}  // namespace rk
