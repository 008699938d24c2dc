// rk_step_tc.cu -- the tensor-core step kernel (rk_step_tc.cuh) of Half
// layers for teams of more than 64 batch rows (one 64-wide k block per
// 128-row tile), the shared-memory plan and the entry point.
#include "rk_step_tc.cuh"

namespace rk {

cudaError_t step_tc_rows(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16,
                         const CUtensorMap* ta, const CUtensorMap* tb) {
  return step_tc_mode_dispatch<0, __half>(p, plan, s, resident, h16, ta, tb);
}

size_t step_tc_smem(int G, int H, int stages, int units) { return tc_smem_layout(G, H, stages, units).total; }

int step_tc_stages(int G, int H, int units, size_t smem_cap) {
  for (int st = SMAXST; st >= 2; --st)
    if (tc_smem_layout(G, H, st, units).total <= smem_cap) return st;
  return 0;
}

cudaError_t step_tc_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16,
                          const CUtensorMap* ta, const CUtensorMap* tb) {
  // 16 rows per direction: the small-batch kernel; 32 units per CTA: a
  // cluster team; else the plan pads a team's rows to 64 (two k blocks per
  // tile) or 128
  if (plan.nbc == 16) return step_tcs_entry(p, plan, s, resident, h16);
  if (p.dtype == 2) {
    __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h16);
    if (plan.J == SJC) return step_tc_cluster(p, plan, s, resident, hp);
    return plan.nbc == 64 ? step_tc_pairs(p, plan, s, resident, hp, ta, tb) : step_tc_rows(p, plan, s, resident, hp, ta, tb);
  }
  __half* hp = static_cast<__half*>(h16);
  if (plan.J == SJC) return step_tc_cluster(p, plan, s, resident, hp);
  return plan.nbc == 64 ? step_tc_pairs(p, plan, s, resident, hp, ta, tb) : step_tc_rows(p, plan, s, resident, hp, ta, tb);
}

}  // namespace rk
