// rk_step_launch.cuh -- picks the step-kernel instantiation for a plan,
// opts it into its shared memory / cluster size and launches it (cluster
// launch for kStepCluster, cooperative launch for kStepGrid).  Included by
// one translation unit per (cell, exchange kind) so they compile in parallel.
#pragma once

#include "rk_step.cuh"

namespace rk {

template <int CELL, typename T, bool GEN, int RPW, int NBC, bool GRID>
cudaError_t step_launch_one(const StepParams& p, const StepPlan& plan, cudaStream_t stream, int* resident_teams) {
  auto kern = step_kernel<CELL, T, GEN, RPW, NBC, GRID>;
  if (plan.threads > MaxThreads<RPW, NBC, GRID>::value || plan.threads % 32 != 0) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  if (!GRID && plan.team_ctas > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if (!GRID) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.team_ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the projection runs; waits for it before reading Xw
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (!GRID && resident_teams == nullptr) ? 2 : 1;
  if (resident_teams != nullptr) {
    if (!GRID) {
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      *resident_teams = (e == cudaSuccess) ? n : 0;
    } else {
      int per_sm = 0, dev = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, plan.threads, plan.smem);
      if (e == cudaSuccess) e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      *resident_teams = (e == cudaSuccess) ? (per_sm * sms) / plan.team_ctas : 0;
    }
    return e;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CELL, typename T, bool GEN, bool GRID>
cudaError_t step_launch_shape(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  switch (plan.shape) {
    case kShapeR8B1:
      if constexpr (!GRID) return step_launch_one<CELL, T, GEN, 8, 1, GRID>(p, plan, s, q);
      break;
    case kShapeR4B8:
      return step_launch_one<CELL, T, GEN, 4, 8, GRID>(p, plan, s, q);
    case kShapeR8B4:
      if constexpr (GRID) return step_launch_one<CELL, T, GEN, 8, 4, GRID>(p, plan, s, q);
      break;
    case kShapeR4B4:
      if constexpr (GRID) return step_launch_one<CELL, T, GEN, 4, 4, GRID>(p, plan, s, q);
      break;
  }
  return cudaErrorInvalidConfiguration;
}

template <int CELL, bool GRID>
cudaError_t step_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  const bool gen = p.generic_acts != 0;
  if (p.dtype == 0) {
    return gen ? step_launch_shape<CELL, float, true, GRID>(p, plan, s, q)
               : step_launch_shape<CELL, float, false, GRID>(p, plan, s, q);
  }
  if (p.dtype == 2) {
    return gen ? step_launch_shape<CELL, __nv_bfloat16, true, GRID>(p, plan, s, q)
               : step_launch_shape<CELL, __nv_bfloat16, false, GRID>(p, plan, s, q);
  }
  return gen ? step_launch_shape<CELL, __half, true, GRID>(p, plan, s, q)
             : step_launch_shape<CELL, __half, false, GRID>(p, plan, s, q);
}

}  // namespace rk
