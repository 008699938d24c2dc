// rk_internal.h -- structures shared between the host side of the library
// (validation, planning, scratch) and the CUDA kernels.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace rk {

constexpr int kMaxActs = 6;
constexpr int kKChunk = 128;      // k is padded to a multiple of 32 lanes x 4 floats
constexpr int kStateHeader = 256; // floats reserved at the start of the state scratch
// 128-row tiles of Xw per direction in the ring the tensor-core step kernel
// uses when it computes the projection itself (16 MB per direction at
// 4096 columns: it stays in L2)
constexpr int kXwRingTiles = 8;
// Region counters of the tensor-core step kernel's teams (16 units per CTA):
// lines of 32 words per team, one per region of 128 k, placed at the start of
// the state scratch's exchange area and zeroed before each launch.
constexpr int kTcRegionLines = 32;
// Counters of the grid step kernel: per team one for h and one for r.h (GRU,
// linear_before_reset = 0), each on a line of 32 words of its own, placed
// after the state header and zeroed before each launch.
constexpr int kGridCounterWordsPerTeam = 2 * 32;

struct ActSlot {
  int kind;
  float alpha, beta;
};

// Which persistent step kernel runs the recurrence.
enum StepKind : int {
  kStepCluster = 0,      // a team is one thread-block cluster; h exchanged through DSMEM
  kStepGrid = 1,         // a team spans many SMs; h exchanged through L2 and a bounded barrier
  kStepClusterFast = 2,  // one batch row per cluster, R in registers, no CTA-wide barrier
  kStepTensor = 3,       // Half: R . h on tcgen05 tensor cores, teams across the grid
};

// Register tile of the step kernel's R.h product: rows per warp x batch rows.
enum StepShape : int {
  kShapeR8B1 = 0,  // 8 rows x 1 batch row
  kShapeR4B8 = 1,  // 4 rows x 8 batch rows
  kShapeR8B4 = 2,  // 8 rows x 4 batch rows
  kShapeR4B4 = 3,  // 4 rows x 4 batch rows (grid kernel: twice the warps of R8B4 on few rows)
};

struct StepParams {
  // problem
  int cell, dtype, direction, layout;
  int S, N, I, H, D, G;
  int T;               // steps the loop runs (max_length or seq)
  float clip;          // > 0: on
  int input_forget, lbr;
  int generic_acts;    // 0: ONNX defaults compiled in
  ActSlot acts[kMaxActs];
  // operands (element offsets already applied)
  const void* R;
  const void* Bias;    // may be null
  const int* lens;     // may be null
  const void* h0;      // may be null
  const void* c0;      // may be null
  const void* P;       // may be null
  void* Y;             // may be null
  void* Yh;            // may be null
  void* Yc;            // may be null
  const float* xw;     // [D, S*N, G*H]
  // plan
  int team_ctas;       // CTAs per team (cluster size for kStepCluster)
  int J;               // hidden units per CTA
  int KP;              // H padded to a multiple of kKChunk
  int nb;              // batch rows per team
  int teams_per_dir;
  int rows_pad;        // rows of R held per CTA (warps x rows per warp)
  int nbc;             // batch rows per h chunk in shared memory
  int stages;          // kStepTensor: 16 KB stages of the h ring
  // projection computed by the launch's last blocks (tensor-core step kernel
  // with flag-published teams, layout 0)
  int fused;           // 1: blocks >= step_ctas run the projection
  int step_ctas;       // blocks of the recurrence
  int pj_M, pj_K;      // X rows (S * N) and input size
  int pj_vec;          // float4 stores of Xw
  int xw_ring;         // tensor-core kernel: Xw ring of this many 128-row tiles per direction (0: whole Xw)
  int xw_consumers;    // warps that signal each step's Xw loads, per direction
  unsigned* xw_done;   // [D]: Xw loads signalled (ring slots are reused once every warp is past them)
  int xw_groups;       // readiness counters per direction
  int xw_mpg;          // 128-row tiles of Xw per counter
  unsigned* xw_ready;  // [D][xw_groups]; 4 per (tile, 256 columns) stored
  // grid exchange (kStepGrid) and status
  float* hglob;        // [2][D*N][KP]
  float* rhglob;       // [D*N][KP]
  unsigned* counters;  // one per team, zero at launch
  unsigned* team_ctrs; // kStepGrid: [teams][2][32] release counters of h and r.h, zero at launch
  int* status;         // device status word (bit 1: timeout)
  long long timeout_ns;
};

struct ProjParams {
  int M, N, K, D;      // Xw[d] (M x N) = X (M x K) . W[d]^T (W[d] is N x K)
  const void* X;
  const void* W;
  float* Xw;
  int dtype;
  int sms;             // SMs of the device (0: queried at launch)
};

struct StepPlan {
  StepKind kind;
  StepShape shape;
  int threads;
  int team_ctas, J, KP, nb, teams_per_dir, rows_pad, nbc;
  int stages;  // kStepTensor: 16 KB stages of the h ring
  size_t smem;
  int grid;
  int kv;     // kStepClusterFast: KP / kKChunk (R chunks per lane and row)
};

// Launchers (defined in the .cu files).  Each returns a cudaError_t.
cudaError_t launch_projection_simt(const ProjParams& p, cudaStream_t s);
// Half projection on tcgen05 tensor cores; cudaErrorNotSupported when the
// operands do not meet its alignment rules (then the SIMT kernel runs).
bool projection_tc_supported(const ProjParams& p);
cudaError_t launch_projection_tc(const ProjParams& p, int* status, long long timeout_ns, cudaStream_t s);
// Tensor maps of X and W for the tcgen05 projection (false if they cannot be
// encoded), and its dynamic shared memory per CTA.
bool projection_tc_maps(const ProjParams& p, CUtensorMap* a, CUtensorMap* b);
size_t projection_tc_smem();
// Step kernel for one cell and exchange kind.  With resident_teams != nullptr
// nothing is launched: the kernel is opted into the plan's shared memory /
// cluster size and the number of teams that can be resident at once is
// returned through the pointer.
template <int CELL, bool GRID>
cudaError_t step_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident_teams);
// The batch-row-per-cluster step kernel (kStepClusterFast), same contract
// as step_entry.
template <int CELL>
cudaError_t step_fast_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident_teams);
// Dynamic shared memory (bytes) the step kernel needs for a plan.
size_t step_smem_for(const StepParams& p, const StepPlan& plan);
// Fixed scratch of rk_encode_noalloc: floats per GPU, and the device
// addresses of the array and its status word for the current device (taken
// with cudaGetSymbolAddress on the first call for each device).
constexpr long long kNoAllocScratchFloats = 4LL << 20;  // 16 MiB
cudaError_t noalloc_scratch(float** scratch, int** status);
// Tensor-core step kernel (kStepTensor): dynamic shared memory for G gates,
// hidden H, `units` hidden units per CTA (16, or 32 for a team that is one
// cluster) and a ring of `stages` 16 KB stages; the most stages (2..8) that
// fit in smem_cap bytes (0 if not even 2 fit); and the launch (resident !=
// nullptr: occupancy query only: co-resident teams, or clusters for a
// cluster team).  h16 is the 16-bit copy of the exchanged hidden state,
// 2 x D x teams x 16 KB regions per 128 k (in the state scratch).
size_t step_tc_smem(int G, int H, int stages, int units);
// Small-batch variant (at most 16 rows per direction, one cluster of
// ceil(H / 32) CTAs per direction; plans it with nbc = 16): dynamic shared
// memory and the launch, same contract as step_tc_entry (its exchanged h
// stays in the CTAs' shared memory: h16 is not used).
size_t step_tcs_smem(int G, int H, bool stacked);
cudaError_t step_tcs_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16);
int step_tc_stages(int G, int H, int units, size_t smem_cap);
cudaError_t step_tc_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16,
                          const CUtensorMap* tmA = nullptr, const CUtensorMap* tmB = nullptr);
// Self-test of the bounded waits (see rk_selftest_timeout).
cudaError_t launch_selftest_timeout(unsigned* counter, int* status, long long timeout_ns, cudaStream_t s);

}  // namespace rk
