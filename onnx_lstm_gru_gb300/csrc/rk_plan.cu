// rk_plan.cu -- shared-memory size of a step-kernel plan (computed from the
// same layout function the kernel uses to carve its shared memory), and the
// self-test of the step kernels' bounded waits.
#include "rk_step.cuh"
#include "rk_step_fast.cuh"

namespace rk {

size_t step_smem_for(const StepParams& p, const StepPlan& plan) {
  if (plan.kind == kStepClusterFast) return fast_smem_layout(p).total;
  const bool grid = plan.kind == kStepGrid;
  const int eb = p.dtype == 0 ? 4 : 2;
  const int nb_ld = grid ? ((plan.nb + plan.nbc - 1) / plan.nbc) * plan.nbc : plan.nbc;  // as in the kernel
  return smem_layout(p, plan.rows_pad, plan.nbc, nb_ld, grid, eb).total;
}

// One CTA waits on a region counter that can never reach its target and on
// an mbarrier phase that nothing completes.  Both waits are the ones the
// step kernels use; each must give up after timeout_ns and set the status.
__global__ void selftest_timeout_kernel(unsigned* counter, int* status, long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  // the counter must reach 1 but nothing raises it
  if (threadIdx.x == 0 && !counter_wait_bounded(counter, 1u, timeout_ns)) atomicOr(status, 1);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // phase 0 needs one arrival that never comes
  if (!mbar_wait_bounded(smem_u32(&bar), 0u, timeout_ns) && threadIdx.x == 0) atomicOr(status, 2);
}

cudaError_t launch_selftest_timeout(unsigned* counter, int* status, long long timeout_ns, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(counter, status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace rk
