// rk_api.cpp -- host side of the C ABI declared in include/rk.h: argument
// checks in 64-bit arithmetic, the launch plan, scratch management and the
// two launches of a layer (projection, then the persistent step kernel).
//
// Behaviour follows the web page "Recurrent layers" (onegpu docs): the
// "Scratch" paragraph (XwLength / StateLength floats, library-owned and grown
// on demand or caller-placed with element offsets; sizes, offsets and shapes
// checked in safe arithmetic before anything is recorded, errors naming
// LSTM/GRU/RNN and the argument) and section "Semantics" (Batch = 0 records
// nothing; Seq = 0 returns the initial states; peepholes, input_forget,
// initial_c and Y_c only for an LSTM, linear_before_reset only for a GRU).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <string>

#include "rk.h"
#include "rk_internal.h"

struct rk_handle {
  uint32_t flags = 0;
  std::string last_error;
  uint64_t launches = 0;
  long long timeout_ns = 2000000000LL;  // 2 s
  bool dev_ready = false;
  int device = -1;
  int sms = 152;
  int smem_optin = 232448;
  int* status = nullptr;
  // status word of the fixed array rk_encode_noalloc last used (device
  // address; null until that entry point has run on this handle)
  int* noalloc_status = nullptr;
  float* xw = nullptr;
  size_t xw_cap = 0;
  float* state = nullptr;
  size_t state_cap = 0;
  unsigned char* host_arena = nullptr;  // device buffers for rk_encode_host
  size_t host_arena_cap = 0;
  bool profiling = false;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};  // proj start/end, step start/end
  bool ev_proj = false, ev_step = false;
  // rk_encode_host: a second stream copies X and the (pageable) operands only
  // the step kernel reads while the first copies W and runs the projection
  cudaStream_t copy_stream = nullptr;
  // fork from the caller's stream; join before the step; X copied (join before the projection)
  cudaEvent_t copy_ev[3] = {nullptr, nullptr, nullptr};
  bool can_map_host = false;  // the device can address page-locked host memory
  // Plans of the last problems encoded (the planner's occupancy queries cost
  // more host time than a small layer takes on the GPU)
  struct PlanEntry {
    bool valid = false;
    rk_problem key;
    uint32_t flags = 0;
    int device = -1;
    rk::StepParams sp;
    rk::StepPlan pl;
  };
  PlanEntry plans[4];
  int plan_next = 0;
};

namespace {

using rk::StepPlan;
using rk::StepParams;

const char* cell_name(int32_t c) {
  switch (c) {
    case RK_LSTM: return "LSTM";
    case RK_GRU: return "GRU";
    case RK_RNN: return "RNN";
    default: return "recurrent";
  }
}

rk_status fail(rk_handle* h, rk_status code, const char* fmt, ...) {
  if (h != nullptr) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    h->last_error = buf;
  }
  return code;
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

int gates_of(int32_t cell) { return cell == RK_LSTM ? 4 : (cell == RK_GRU ? 3 : 1); }
int acts_per_dir(int32_t cell) { return cell == RK_LSTM ? 3 : (cell == RK_GRU ? 2 : 1); }
int dirs_of(const rk_problem* p) { return p->direction == RK_BIDIRECTIONAL ? 2 : 1; }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Element counts of every operand; -1 where a product overflows.
struct Extents {
  int64_t X, W, R, B, lens, state, P, Y;
};

bool extents_of(const rk_problem* p, Extents* e) {
  const int64_t G = gates_of(p->cell), D = dirs_of(p);
  int64_t GH, t1, t2;
  if (!mul_ok(G, p->hidden, &GH)) return false;
  if (!mul_ok(p->seq, p->batch, &t1) || !mul_ok(t1, p->input, &e->X)) return false;
  if (!mul_ok(D, GH, &t1) || !mul_ok(t1, p->input, &e->W)) return false;
  if (!mul_ok(t1, p->hidden, &e->R)) return false;
  if (!mul_ok(t1, 2, &e->B)) return false;
  e->lens = p->batch;
  if (!mul_ok(D, p->batch, &t2) || !mul_ok(t2, p->hidden, &e->state)) return false;
  if (!mul_ok(D, 3, &t1) || !mul_ok(t1, p->hidden, &e->P)) return false;
  if (!mul_ok(p->seq, e->state, &e->Y)) return false;
  return true;
}

rk_status check_tensor(rk_handle* h, const rk_problem* p, const char* name, const rk_tensor& t, int64_t extent,
                       bool required) {
  const char* cn = cell_name(p->cell);
  if (t.ptr == nullptr) {
    if (required && extent > 0) return fail(h, RK_ERR_SHAPE, "%s: %s: required tensor is null", cn, name);
    return RK_OK;
  }
  if (t.offset < 0) return fail(h, RK_ERR_SHAPE, "%s: %s: negative offset %lld", cn, name, (long long)t.offset);
  if (t.length < 0) return fail(h, RK_ERR_SHAPE, "%s: %s: negative length %lld", cn, name, (long long)t.length);
  int64_t end;
  if (!add_ok(t.offset, extent, &end))
    return fail(h, RK_ERR_SHAPE, "%s: %s: offset %lld + extent %lld overflows", cn, name, (long long)t.offset,
                (long long)extent);
  if (end > t.length)
    return fail(h, RK_ERR_SHAPE, "%s: %s: offset %lld + extent %lld exceeds buffer length %lld", cn, name,
                (long long)t.offset, (long long)extent, (long long)t.length);
  return RK_OK;
}

rk_status validate_problem(rk_handle* h, const rk_problem* p) {
  if (p == nullptr) return fail(h, RK_ERR_ARG, "recurrent: problem is null");
  if (p->cell < RK_LSTM || p->cell > RK_RNN) return fail(h, RK_ERR_SHAPE, "recurrent: cell: unknown value %d", p->cell);
  const char* cn = cell_name(p->cell);
  if (p->direction < RK_FORWARD || p->direction > RK_BIDIRECTIONAL)
    return fail(h, RK_ERR_SHAPE, "%s: direction: unknown value %d", cn, p->direction);
  if (p->dtype != RK_F32 && p->dtype != RK_F16 && p->dtype != RK_BF16)
    return fail(h, RK_ERR_SHAPE, "%s: dtype: unknown value %d", cn, p->dtype);
  if (p->layout != 0 && p->layout != 1) return fail(h, RK_ERR_SHAPE, "%s: layout: must be 0 or 1, got %d", cn, p->layout);
  const int64_t lim = 0x7fffffffLL;
  if (p->seq < 0 || p->seq > lim) return fail(h, RK_ERR_SHAPE, "%s: seq: %lld out of range", cn, (long long)p->seq);
  if (p->batch < 0 || p->batch > lim)
    return fail(h, RK_ERR_SHAPE, "%s: batch: %lld out of range", cn, (long long)p->batch);
  if (p->input < 0 || p->input > lim)
    return fail(h, RK_ERR_SHAPE, "%s: input: %lld out of range", cn, (long long)p->input);
  if (p->hidden < 0 || p->hidden > lim)
    return fail(h, RK_ERR_SHAPE, "%s: hidden: %lld out of range", cn, (long long)p->hidden);
  if (p->input_forget != 0 && p->cell != RK_LSTM)
    return fail(h, RK_ERR_SHAPE, "%s: input_forget: only an LSTM has it", cn);
  if (p->linear_before_reset != 0 && p->cell != RK_GRU)
    return fail(h, RK_ERR_SHAPE, "%s: linear_before_reset: only a GRU has it", cn);
  const int want = acts_per_dir(p->cell) * dirs_of(p);
  if (p->num_acts != 0 && p->num_acts != want)
    return fail(h, RK_ERR_SHAPE, "%s: activations: expected 0 or %d, got %d", cn, want, p->num_acts);
  for (int i = 0; i < p->num_acts; ++i)
    if (p->act[i].kind < RK_ACT_SIGMOID || p->act[i].kind > RK_ACT_SOFTPLUS)
      return fail(h, RK_ERR_SHAPE, "%s: activations[%d]: unknown kind %d", cn, i, p->act[i].kind);
  if (p->max_length < 0 || p->max_length > p->seq)
    return fail(h, RK_ERR_SHAPE, "%s: max_length: %lld not in [0, seq=%lld]", cn, (long long)p->max_length,
                (long long)p->seq);
  Extents e;
  if (!extents_of(p, &e)) return fail(h, RK_ERR_SHAPE, "%s: sizes overflow 64-bit element counts", cn);
  int64_t m, gh;
  if (!mul_ok(p->seq, p->batch, &m) || m > lim || !mul_ok(gates_of(p->cell), p->hidden, &gh) || gh > lim)
    return fail(h, RK_ERR_UNSUPPORTED, "%s: seq*batch or gates*hidden exceeds 2^31 - 1", cn);
  return RK_OK;
}

rk_status validate_all(rk_handle* h, const rk_problem* p, const rk_operands* o) {
  rk_status st = validate_problem(h, p);
  if (st != RK_OK) return st;
  if (o == nullptr) return fail(h, RK_ERR_ARG, "%s: operands: null", cell_name(p->cell));
  const char* cn = cell_name(p->cell);
  Extents e;
  extents_of(p, &e);
  const bool lstm = p->cell == RK_LSTM;
  if (!lstm) {
    if (o->P.ptr) return fail(h, RK_ERR_SHAPE, "%s: P: peepholes exist only for an LSTM", cn);
    if (o->initial_c.ptr) return fail(h, RK_ERR_SHAPE, "%s: initial_c: exists only for an LSTM", cn);
    if (o->Y_c.ptr) return fail(h, RK_ERR_SHAPE, "%s: Y_c: exists only for an LSTM", cn);
  }
  if (p->max_length > 0 && p->max_length < p->seq && o->sequence_lens.ptr == nullptr)
    return fail(h, RK_ERR_SHAPE, "%s: max_length: %lld < seq needs sequence_lens", cn, (long long)p->max_length);
  if ((st = check_tensor(h, p, "X", o->X, e.X, true)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "W", o->W, e.W, true)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "R", o->R, e.R, true)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "B", o->B, e.B, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "sequence_lens", o->sequence_lens, e.lens, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "initial_h", o->initial_h, e.state, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "initial_c", o->initial_c, e.state, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "P", o->P, e.P, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "Y", o->Y, e.Y, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "Y_h", o->Y_h, e.state, false)) != RK_OK) return st;
  if ((st = check_tensor(h, p, "Y_c", o->Y_c, e.state, false)) != RK_OK) return st;
  return RK_OK;
}

int64_t xw_len(const rk_problem* p) {
  if (p->seq == 0 || p->batch == 0) return 0;
  return (int64_t)dirs_of(p) * p->seq * p->batch * gates_of(p->cell) * p->hidden;
}
int64_t kp_of(const rk_problem* p) { return round_up(std::max<int64_t>(p->hidden, 1), rk::kKChunk); }
// Counter words of the grid step kernel (teams of up to 64 batch rows).
int64_t grid_counter_words(const rk_problem* p) {
  return (int64_t)dirs_of(p) * ((p->batch + 63) / 64) * rk::kGridCounterWordsPerTeam;
}
int64_t state_len(const rk_problem* p) {
  // counters, the grid kernel's team counters, the double-buffered float32
  // h of the grid kernel, and a region for r.h (grid kernel) or the 16-bit
  // copies of h (tensor-core kernel)
  return rk::kStateHeader + grid_counter_words(p) + 2 * (int64_t)dirs_of(p) * p->batch * kp_of(p) +
         (int64_t)dirs_of(p) * (p->batch + 128) * kp_of(p);
}

rk_status ensure_device(rk_handle* h) {
  if (h->dev_ready) return RK_OK;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
  int map = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&map, cudaDevAttrCanMapHostMemory, h->device);
  h->can_map_host = map != 0;
  if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int));
  if (e != cudaSuccess) return fail(h, RK_ERR_CUDA, "recurrent: device setup failed: %s", cudaGetErrorName(e));
  h->dev_ready = true;
  return RK_OK;
}

void fill_params_problem(const rk_problem* p, StepParams* sp) {
  std::memset(sp, 0, sizeof(*sp));
  sp->cell = p->cell;
  sp->dtype = p->dtype;
  sp->direction = p->direction;
  sp->layout = p->layout;
  sp->S = (int)p->seq;
  sp->N = (int)p->batch;
  sp->I = (int)p->input;
  sp->H = (int)p->hidden;
  sp->D = dirs_of(p);
  sp->G = gates_of(p->cell);
  sp->T = (int)(p->max_length > 0 ? p->max_length : p->seq);
  sp->clip = p->clip;
  sp->input_forget = p->input_forget != 0;
  sp->lbr = p->linear_before_reset != 0;
  const int want = acts_per_dir(p->cell) * sp->D;
  if (p->num_acts == 0) {
    sp->generic_acts = 0;
    const int defk[3][3] = {{RK_ACT_SIGMOID, RK_ACT_TANH, RK_ACT_TANH}, {RK_ACT_SIGMOID, RK_ACT_TANH, 0}, {RK_ACT_TANH, 0, 0}};
    for (int i = 0; i < want; ++i) sp->acts[i] = {defk[p->cell][i % acts_per_dir(p->cell)], 0.0f, 0.0f};
  } else {
    sp->generic_acts = 1;
    for (int i = 0; i < want; ++i) sp->acts[i] = {p->act[i].kind, p->act[i].alpha, p->act[i].beta};
  }
  sp->KP = (int)kp_of(p);
}

// Whether the tensor-core recurrence computes the projection itself on the
// SMs it leaves idle: flag-published teams (the projection's tiles are
// produced in the order the steps consume them, which needs layout 0), the
// tcgen05 projection usable, at least 8 idle SMs, and room in the state
// header for the readiness counters after the teams' flags.  With maps !=
// nullptr the tensor maps are encoded too (needs the operands).
struct FusedProj {
  bool on = false;
  int np = 0, groups = 0, mpg = 0, counter0 = 0;
};
FusedProj fused_projection(const rk_handle* h, const rk_problem* p, const StepPlan& pl, const rk::ProjParams& pp,
                           bool has_projection, CUtensorMap* tmA, CUtensorMap* tmB) {
  FusedProj f;
  if (!has_projection || pl.kind != rk::kStepTensor || pl.J != 16 || p->layout != 0 || p->dtype == RK_F32 ||
      (h->flags & (RK_FORCE_SIMT_PROJECTION | RK_SEPARATE_PROJECTION)) || p->input % 8 != 0)
    return f;
  const int D = dirs_of(p);
  const int np = h->sms - pl.grid;
  const int counter0 = D * pl.teams_per_dir * ((pl.team_ctas + 7) / 8 * 8);
  // the last D words of the header: the Xw ring's consumption counters
  const int groups = (rk::kStateHeader - counter0 - D) / D;
  const int mt = (pp.M + 127) / 128;
  if (np < 8 || groups < 1 || mt < 1) return f;
  if (tmA != nullptr && !(rk::projection_tc_supported(pp) && rk::projection_tc_maps(pp, tmA, tmB))) return f;
  f.on = true;
  f.np = np;
  f.groups = std::min(groups, mt);
  f.mpg = (mt + f.groups - 1) / f.groups;
  f.counter0 = counter0;
  return f;
}

// Floats at the start of the state scratch that must be zero when the step
// kernel starts: the header (barrier counters, readiness counters), and for
// the tensor-core kernel with teams of 16-unit CTAs its region counters.
int64_t zeroed_state_floats(const StepPlan& pl, int D) {
  int64_t n = rk::kStateHeader;
  if (pl.kind == rk::kStepTensor && pl.J == 16) n += (int64_t)D * pl.teams_per_dir * rk::kTcRegionLines * 32;
  if (pl.kind == rk::kStepGrid) n += (int64_t)D * pl.teams_per_dir * rk::kGridCounterWordsPerTeam;
  return n;
}

// The step kernel's pointers into the state scratch: the header, then (grid
// kernel) its team counters, then the exchange buffers.
void assign_state(rk::StepParams& sp, const StepPlan& pl, float* state) {
  sp.counters = reinterpret_cast<unsigned*>(state);
  float* exchange = state + rk::kStateHeader;
  if (pl.kind == rk::kStepGrid) {
    sp.team_ctrs = reinterpret_cast<unsigned*>(exchange);
    exchange += (size_t)sp.D * pl.teams_per_dir * rk::kGridCounterWordsPerTeam;
  }
  sp.hglob = exchange;
  sp.rhglob = sp.hglob + (size_t)2 * sp.D * sp.N * sp.KP;
}

// Launch (or, with resident != nullptr, size) the step kernel of a plan.
cudaError_t step_dispatch(int32_t cell, const StepParams& sp, const StepPlan& pl, cudaStream_t stream, int* resident) {
  if (pl.kind == rk::kStepTensor) return rk::step_tc_entry(sp, pl, stream, resident, sp.rhglob);
  if (pl.kind == rk::kStepClusterFast) {
    switch (cell) {
      case RK_LSTM: return rk::step_fast_entry<0>(sp, pl, stream, resident);
      case RK_GRU: return rk::step_fast_entry<1>(sp, pl, stream, resident);
      default: return rk::step_fast_entry<2>(sp, pl, stream, resident);
    }
  }
  const bool grid = pl.kind == rk::kStepGrid;
  switch (cell) {
    case RK_LSTM: return grid ? rk::step_entry<0, true>(sp, pl, stream, resident) : rk::step_entry<0, false>(sp, pl, stream, resident);
    case RK_GRU: return grid ? rk::step_entry<1, true>(sp, pl, stream, resident) : rk::step_entry<1, false>(sp, pl, stream, resident);
    default: return grid ? rk::step_entry<2, true>(sp, pl, stream, resident) : rk::step_entry<2, false>(sp, pl, stream, resident);
  }
}

// Step-kernel plan, in order of preference: the one-row-per-cluster
// kernel (R in registers) when a row's hidden units fit 16 CTAs of <= 32
// units, R's chunks fit the registers and every cluster fits the GPU at
// once; else, for 16-bit layers with 4 or more rows, a tensor-core kernel;
// else the cluster kernel when R fits one cluster's shared memory; else the
// grid kernel.  RK_PREFER_TENSOR_STEP puts the tensor-core kernels first.
// `check` asks the occupancy API (needs a device).
rk_status plan_step_uncached(rk_handle* h, const rk_problem* p, StepParams* sp, StepPlan* out, bool check) {
  const int G = sp->G, D = sp->D, N = sp->N, H = sp->H, KP = sp->KP;
  const int eb = p->dtype == RK_F32 ? 4 : 2;
  const bool lbr0 = p->cell == RK_GRU && !p->linear_before_reset;
  (void)lbr0;
  const int smem_cap = h->smem_optin - 1024;  // room for the kernel's static shared memory
  auto finish = [&](StepPlan& pl) -> bool {
    sp->team_ctas = pl.team_ctas;
    sp->J = pl.J;
    sp->nb = pl.nb;
    sp->teams_per_dir = pl.teams_per_dir;
    sp->rows_pad = pl.rows_pad;
    sp->nbc = pl.nbc;
    pl.KP = KP;
    pl.smem = rk::step_smem_for(*sp, pl);
    return pl.smem > 0 && (int)pl.smem <= smem_cap;
  };
  auto resident = [&](const StepPlan& pl) -> int {
    int teams = 0;
    cudaError_t e = step_dispatch(p->cell, *sp, pl, nullptr, &teams);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return teams;
  };
  // fast kernel: one batch row per cluster, R rows in registers.  Largest
  // cluster (<= 16 CTAs) whose clusters all fit the GPU at once, with 16 to
  // 32 hidden units per CTA (fewer when H itself is smaller).  Where it fits
  // it beats the tensor-core kernels at every size measured (16-bit
  // bidirectional layers, H 64 to 512, 4 to 16 rows: 0.7-2.0 against
  // 1.9-3.5 us per step), its h exchange being a push into the peers'
  // shared memory rather than a publication through global memory.
  const int KV = KP / rk::kKChunk;
  const bool kv_ok = (p->dtype == RK_F32 ? KV <= 2 : KV <= 4) && KV != 3;
  const int U = p->cell == RK_RNN ? 8 : (KV <= 2 ? 4 : 2);  // units per warp, as the kernel uses
  auto try_fast = [&]() -> bool {
    if ((h->flags & (RK_FORCE_GRID_STEP | RK_FORCE_GENERAL_STEP)) || !kv_ok) return false;
    for (int C = 16; C >= 1; C /= 2) {
      StepPlan pl{};
      pl.kind = rk::kStepClusterFast;
      pl.shape = rk::kShapeR8B1;
      pl.team_ctas = C;
      pl.J = (H + C - 1) / C;
      if (pl.J > 32 || pl.J < std::min(H, 16)) continue;
      if (C > 1 && (int64_t)(C - 1) * pl.J >= H) continue;  // no CTA without units
      if ((int64_t)D * N * C > h->sms) continue;            // all clusters at once
      pl.nb = 1;
      pl.nbc = 1;
      pl.teams_per_dir = N;
      pl.kv = KV;
      pl.threads = (pl.J + U - 1) / U * 32;
      pl.grid = D * N * C;
      if (!finish(pl)) continue;
      if (check && resident(pl) < 1) continue;
      *out = pl;
      return true;
    }
    return false;
  };
  const bool tensor_first = p->dtype != RK_F32 && (h->flags & RK_PREFER_TENSOR_STEP);
  if (!tensor_first && try_fast()) return RK_OK;
  // tensor-core kernel: 16-bit layers (Half or bfloat16) with a batch worth
  // a dense product (R . h on tcgen05), every CTA of the launch resident at once
  if (p->dtype != RK_F32 && !(h->flags & (RK_FORCE_GRID_STEP | RK_FORCE_GENERAL_STEP | RK_FORCE_SIMT_STEP)) &&
      H % 8 == 0 && N >= 4) {
    // at most 16 rows per direction: the gate rows are the MMA's M and the
    // batch its N, one cluster of ceil(H / 32) CTAs per direction
    const int Cc = (H + 31) / 32;
    if (N <= 16 && Cc <= 16) {
      StepPlan pl{};
      pl.kind = rk::kStepTensor;
      pl.team_ctas = Cc;
      pl.nb = N;
      pl.nbc = 16;
      pl.teams_per_dir = 1;
      pl.J = 32;
      pl.threads = 320;
      pl.grid = D * Cc;
      pl.stages = 1;
      pl.smem = rk::step_tcs_smem(G, H, (p->cell == RK_GRU && !p->linear_before_reset) || p->cell == RK_RNN);
      if ((int)pl.smem <= smem_cap && (!check || resident(pl) >= 1)) {
        sp->team_ctas = pl.team_ctas;
        sp->J = pl.J;
        sp->nb = pl.nb;
        sp->teams_per_dir = pl.teams_per_dir;
        sp->nbc = pl.nbc;
        sp->stages = pl.stages;
        *out = pl;
        return RK_OK;
      }
    }
    // (GRU with linear_before_reset = 0 needs r (.) h exchanged within the
    // step: only the small-batch kernel does that on the tensor cores)
    const bool lbr0_cell = p->cell == RK_GRU && !p->linear_before_reset;
    // a team of at most 64 rows whose units fit one cluster at 32 per CTA
    // publishes h inside the cluster (remote mbarrier arrivals), far faster
    // than global flags; teams never wait on each other
    if (!lbr0_cell && N <= 64 && Cc <= 16 && (H + 63) / 64 <= 32) {
      StepPlan pl{};
      pl.kind = rk::kStepTensor;
      pl.team_ctas = Cc;
      pl.nb = N;
      pl.nbc = 64;
      pl.teams_per_dir = 1;
      pl.J = 32;
      pl.threads = 320;
      pl.grid = D * Cc;
      pl.stages = rk::step_tc_stages(G, H, 32, (size_t)smem_cap);
      pl.smem = rk::step_tc_smem(G, H, std::max(pl.stages, 2), 32);
      if (pl.stages >= 2 && (!check || resident(pl) >= 1)) {
        sp->team_ctas = pl.team_ctas;
        sp->J = pl.J;
        sp->nb = pl.nb;
        sp->teams_per_dir = pl.teams_per_dir;
        sp->nbc = pl.nbc;
        sp->stages = pl.stages;
        *out = pl;
        return RK_OK;
      }
    }
    StepPlan pl{};
    pl.kind = rk::kStepTensor;
    pl.team_ctas = (H + 15) / 16;
    pl.nb = std::min(N, 128);
    // rows of h per 128 k: a team of at most 64 rows pairs two 64-wide k
    // blocks in one 128-row tile
    pl.nbc = pl.nb <= 64 ? 64 : 128;
    pl.teams_per_dir = (N + 127) / 128;
    pl.J = 16;
    pl.threads = 320;
    pl.grid = D * pl.teams_per_dir * pl.team_ctas;
    pl.stages = rk::step_tc_stages(G, H, 16, (size_t)smem_cap);
    pl.smem = rk::step_tc_smem(G, H, std::max(pl.stages, 2), 16);
    // one publication flag per CTA in the state header, each team's starting
    // on a 32-byte boundary; one polling lane per 128 k
    const int teams = D * pl.teams_per_dir;
    const bool fits = !lbr0_cell && pl.stages >= 2 && pl.grid <= h->sms &&
                      teams * ((pl.team_ctas + 7) / 8 * 8) <= rk::kStateHeader && (H + 63) / 64 <= 32;
    if (fits && (!check || resident(pl) * pl.team_ctas >= pl.grid)) {
      sp->team_ctas = pl.team_ctas;
      sp->J = pl.J;
      sp->nb = pl.nb;
      sp->teams_per_dir = pl.teams_per_dir;
      sp->nbc = pl.nbc;
      sp->stages = pl.stages;
      *out = pl;
      return RK_OK;
    }
  }
  if (tensor_first && try_fast()) return RK_OK;
  if (!(h->flags & RK_FORCE_GRID_STEP)) {
    const int nb = N == 1 ? 1 : std::min(N, 8);
    const rk::StepShape shape = nb == 1 ? rk::kShapeR8B1 : rk::kShapeR4B8;
    const int rpw = shape == rk::kShapeR8B1 ? 8 : 4;
    const int maxt = shape == rk::kShapeR8B1 ? 512 : 768;
    for (int C = 1; C <= 16; C *= 2) {
      StepPlan pl{};
      pl.kind = rk::kStepCluster;
      pl.shape = shape;
      pl.team_ctas = C;
      pl.J = (int)((H + C - 1) / C);
      pl.nb = nb;
      pl.nbc = nb == 1 ? 1 : 8;
      pl.teams_per_dir = (N + nb - 1) / nb;
      const int Jp = (int)round_up(pl.J, rpw);
      pl.rows_pad = G * Jp;
      const int warps = pl.rows_pad / rpw;
      pl.threads = (int)std::max<int64_t>(32 * warps, round_up((int64_t)pl.J * nb, 32));
      pl.threads = std::max(pl.threads, 64);
      pl.grid = D * pl.teams_per_dir * C;
      const int64_t rbytes = (int64_t)pl.rows_pad * KP * eb;
      if (pl.threads > maxt) continue;
      if (rbytes > 64 * 1024 && C < 16) continue;  // spread R until a slice is <= 64 KB
      if (!finish(pl)) continue;
      if (check && resident(pl) < 1) continue;
      *out = pl;
      return RK_OK;
    }
  }
  // grid kernel: all SMs, one CTA each, teams of up to 64 batch rows
  {
    StepPlan pl{};
    pl.kind = rk::kStepGrid;
    const int nb = std::min(N, 64);
    pl.nb = nb;
    pl.teams_per_dir = (N + nb - 1) / nb;
    pl.nbc = nb <= 4 ? 4 : 8;
    const int teams = D * pl.teams_per_dir;
    if (teams > rk::kStateHeader)
      return fail(h, RK_ERR_UNSUPPORTED, "%s: batch %d needs too many grid teams", cell_name(p->cell), N);
    int per_team = h->sms / teams;
    if (per_team < 1)
      return fail(h, RK_ERR_UNSUPPORTED, "%s: %d teams exceed %d SMs", cell_name(p->cell), teams, h->sms);
    pl.J = (H + per_team - 1) / per_team;
    pl.team_ctas = (H + pl.J - 1) / pl.J;
    // up to 4 batch rows: 8-row register tiles, or 4-row ones when 8-row
    // tiles would leave warps of a 256-thread block without rows
    pl.shape = nb <= 4 ? (G * round_up(pl.J, 8) / 8 < 8 ? rk::kShapeR4B4 : rk::kShapeR8B4) : rk::kShapeR4B8;
    const int rpw = pl.shape == rk::kShapeR8B4 ? 8 : 4;
    const int Jp = (int)round_up(pl.J, rpw);
    pl.rows_pad = G * Jp;
    // computing warps (a warp per row group, up to the kernel's thread
    // budget) and one warp that stages the exchanged rows
    const int max_threads = pl.shape == rk::kShapeR4B4 ? 320 : 640;
    pl.threads = (int)std::min<int64_t>(max_threads - 32, std::max<int64_t>(256, 32 * (pl.rows_pad / rpw))) + 32;
    pl.grid = teams * pl.team_ctas;
    if (!finish(pl))
      return fail(h, RK_ERR_UNSUPPORTED, "%s: R slice of %d rows x %d does not fit shared memory", cell_name(p->cell),
                  pl.rows_pad, KP);
    if (check) {
      // every CTA of the launch must be resident at once
      const int r = resident(pl);
      if (r * pl.team_ctas < pl.grid)
        return fail(h, RK_ERR_UNSUPPORTED, "%s: grid step kernel needs %d co-resident CTAs", cell_name(p->cell), pl.grid);
    }
    *out = pl;
    return RK_OK;
  }
}

// The problem's fields alone (no padding bytes, which the caller may leave
// uninitialised), for comparing problems byte by byte.
rk_problem plan_key(const rk_problem* p) {
  rk_problem k;
  std::memset(&k, 0, sizeof(k));
  k.cell = p->cell;
  k.direction = p->direction;
  k.dtype = p->dtype;
  k.layout = p->layout;
  k.seq = p->seq;
  k.batch = p->batch;
  k.input = p->input;
  k.hidden = p->hidden;
  k.clip = p->clip;
  k.input_forget = p->input_forget;
  k.linear_before_reset = p->linear_before_reset;
  k.num_acts = p->num_acts;
  for (int i = 0; i < 6; ++i) k.act[i] = p->act[i];
  k.max_length = p->max_length;
  return k;
}

// plan_step_uncached, remembered per handle: with check set the plan of a
// problem depends only on its fields, the handle's flags and the device, so
// a problem seen before takes its plan (and the step parameters the planner
// filled) from the handle instead of repeating the occupancy queries.
rk_status plan_step(rk_handle* h, const rk_problem* p, StepParams* sp, StepPlan* out, bool check) {
  if (!check) return plan_step_uncached(h, p, sp, out, check);
  const rk_problem key = plan_key(p);
  for (const auto& e : h->plans) {
    if (e.valid && e.flags == h->flags && e.device == h->device && std::memcmp(&e.key, &key, sizeof(key)) == 0) {
      *sp = e.sp;
      *out = e.pl;
      return RK_OK;
    }
  }
  const rk_status st = plan_step_uncached(h, p, sp, out, check);
  if (st == RK_OK) {
    auto& e = h->plans[h->plan_next];
    h->plan_next = (h->plan_next + 1) % 4;
    e.valid = true;
    e.key = key;
    e.flags = h->flags;
    e.device = h->device;
    e.sp = *sp;
    e.pl = *out;
  }
  return st;
}

rk_status cuda_fail(rk_handle* h, const rk_problem* p, const char* what, cudaError_t e) {
  return fail(h, RK_ERR_CUDA, "%s: %s: %s (%s)", cell_name(p->cell), what, cudaGetErrorName(e), cudaGetErrorString(e));
}

rk_status grow(rk_handle* h, float** buf, size_t* cap, size_t need, const rk_problem* p, const char* what) {
  if (*cap >= need) return RK_OK;
  if (*buf) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, p, what, e);
    cudaFree(*buf);
    *buf = nullptr;
    *cap = 0;
  }
  cudaError_t e = cudaMalloc(buf, need * sizeof(float));
  if (e != cudaSuccess) {
    cudaGetLastError();
    *buf = nullptr;
    return fail(h, RK_ERR_OOM, "%s: %s: cannot allocate %zu bytes of scratch", cell_name(p->cell), what,
                need * sizeof(float));
  }
  *cap = need;
  return RK_OK;
}

const void* tptr(const rk_tensor& t, int eb) {
  return t.ptr ? static_cast<const void*>(static_cast<const char*>(t.ptr) + t.offset * eb) : nullptr;
}
void* tptr_mut(const rk_tensor& t, int eb) {
  return t.ptr ? static_cast<void*>(static_cast<char*>(t.ptr) + t.offset * eb) : nullptr;
}

}  // namespace

extern "C" {

int32_t rk_version(void) { return 100; }

rk_status rk_create(rk_handle** out, uint32_t flags) {
  if (out == nullptr) return RK_ERR_ARG;
  *out = new (std::nothrow) rk_handle();
  if (*out == nullptr) return RK_ERR_OOM;
  (*out)->flags = flags;
  return RK_OK;
}

rk_status rk_destroy(rk_handle* h) {
  if (h == nullptr) return RK_OK;
  if (h->dev_ready) {
    cudaDeviceSynchronize();
    for (auto& ev : h->ev)
      if (ev) cudaEventDestroy(ev);
    for (auto& ev : h->copy_ev)
      if (ev) cudaEventDestroy(ev);
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    cudaFree(h->status);
    cudaFree(h->xw);
    cudaFree(h->state);
    cudaFree(h->host_arena);
  }
  delete h;
  return RK_OK;
}

int64_t rk_xw_length(const rk_problem* p) {
  if (validate_problem(nullptr, p) != RK_OK) return -1;
  return xw_len(p);
}

int64_t rk_state_length(const rk_problem* p) {
  if (validate_problem(nullptr, p) != RK_OK) return -1;
  return state_len(p);
}

rk_status rk_validate(rk_handle* h, const rk_problem* p, const rk_operands* ops) {
  if (h == nullptr) return RK_ERR_ARG;
  h->last_error.clear();
  return validate_all(h, p, ops);
}

rk_status rk_validate_lengths(rk_handle* h, const rk_problem* p, const int32_t* lens, int64_t n) {
  if (h == nullptr || p == nullptr) return RK_ERR_ARG;
  h->last_error.clear();
  rk_status st = validate_problem(h, p);
  if (st != RK_OK) return st;
  if (n > 0 && lens == nullptr) return fail(h, RK_ERR_ARG, "%s: sequence_lens: null host pointer", cell_name(p->cell));
  if (n != p->batch)
    return fail(h, RK_ERR_SHAPE, "%s: sequence_lens: %lld values for batch %lld", cell_name(p->cell), (long long)n,
                (long long)p->batch);
  const int64_t hi = p->max_length > 0 ? std::min<int64_t>(p->max_length, p->seq) : p->seq;
  for (int64_t b = 0; b < n; ++b) {
    if (lens[b] < 0 || lens[b] > hi)
      return fail(h, RK_ERR_SHAPE, "%s: sequence_lens[%lld] = %d outside [0, %lld]%s", cell_name(p->cell),
                  (long long)b, (int)lens[b], (long long)hi, p->max_length > 0 ? " (max_length)" : " (seq)");
  }
  return RK_OK;
}

rk_status rk_describe_plan(rk_handle* h, const rk_problem* p, char* buf, int64_t len) {
  if (h == nullptr || buf == nullptr || len <= 0) return RK_ERR_ARG;
  rk_status st = validate_problem(h, p);
  if (st != RK_OK) return st;
  StepParams sp;
  fill_params_problem(p, &sp);
  StepPlan pl{};
  int dev = 0;
  const bool have_dev = cudaGetDevice(&dev) == cudaSuccess;
  if (!have_dev) cudaGetLastError();
  if (have_dev) {
    if ((st = ensure_device(h)) != RK_OK) return st;
  }
  if (p->batch == 0 || p->hidden == 0) {
    snprintf(buf, (size_t)len, "noop");
    return RK_OK;
  }
  if ((st = plan_step(h, p, &sp, &pl, have_dev)) != RK_OK) return st;
  const bool tc = p->dtype != RK_F32 && !(h->flags & RK_FORCE_SIMT_PROJECTION) && p->input > 0 && p->input % 8 == 0;
  rk::ProjParams pp{};
  pp.M = (int)(p->seq * p->batch);
  const bool fused = fused_projection(h, p, pl, pp, p->seq > 0 && p->input > 0, nullptr, nullptr).on;
  snprintf(buf, (size_t)len, "proj=%s step=%s shape=%d ctas=%d J=%d nb=%d teams=%d threads=%d smem=%zu grid=%d",
           fused ? "fused" : (tc ? "tc" : "simt"),
           pl.kind == rk::kStepTensor ? "tensor"
                                      : (pl.kind == rk::kStepClusterFast ? "fast" : (pl.kind == rk::kStepCluster ? "cluster" : "grid")),
           (int)pl.shape, pl.team_ctas, pl.J, pl.nb, pl.teams_per_dir * sp.D, pl.threads, pl.smem, pl.grid);
  if (pl.kind == rk::kStepTensor) {
    // which tensor-core kernel: small batch (gate rows as M), cluster team,
    // or flag-published teams with paired / single k blocks per tile
    const char* v = pl.nbc == 16 ? "small" : (pl.J == 32 ? "cluster" : (pl.nbc == 64 ? "pairs" : "rows"));
    const size_t n = strlen(buf);
    if (n + 1 < (size_t)len) snprintf(buf + n, (size_t)len - n, " variant=%s", v);
  }
  return RK_OK;
}

namespace {

// The layer on validated operands.  step_wait != nullptr: the stream waits
// for that event just before the step kernel's launch (the host entry's
// copies of the operands only the step kernel reads).
rk_status encode_validated(rk_handle* h, const rk_problem* p, const rk_operands* ops, const rk_scratch* scratch,
                           cudaStream_t stream, cudaEvent_t step_wait) {
  rk_status st;
  const int eb = p->dtype == RK_F32 ? 4 : 2;

  StepParams sp;
  fill_params_problem(p, &sp);
  StepPlan pl{};
  if ((st = plan_step(h, p, &sp, &pl, true)) != RK_OK) return st;

  // scratch: caller-placed or grown on demand
  const int64_t need_xw = xw_len(p), need_state = state_len(p);
  float* xw = nullptr;
  float* state = nullptr;
  if (scratch != nullptr && scratch->xw != nullptr) {
    if (scratch->xw_offset < 0 || scratch->xw_offset > scratch->xw_length ||
        scratch->xw_length - scratch->xw_offset < need_xw)
      return fail(h, RK_ERR_SHAPE, "%s: xw scratch: offset %lld + %lld floats exceeds length %lld", cell_name(p->cell),
                  (long long)scratch->xw_offset, (long long)need_xw, (long long)scratch->xw_length);
    xw = scratch->xw + scratch->xw_offset;
  } else {
    if ((st = grow(h, &h->xw, &h->xw_cap, (size_t)std::max<int64_t>(need_xw, 1), p, "xw scratch")) != RK_OK) return st;
    xw = h->xw;
  }
  if (scratch != nullptr && scratch->state != nullptr) {
    if (scratch->state_offset < 0 || scratch->state_offset > scratch->state_length ||
        scratch->state_length - scratch->state_offset < need_state)
      return fail(h, RK_ERR_SHAPE, "%s: state scratch: offset %lld + %lld floats exceeds length %lld",
                  cell_name(p->cell), (long long)scratch->state_offset, (long long)need_state,
                  (long long)scratch->state_length);
    state = scratch->state + scratch->state_offset;
    if (reinterpret_cast<uintptr_t>(state) % 16 != 0)
      return fail(h, RK_ERR_SHAPE, "%s: state scratch: base + offset must be 16-byte aligned", cell_name(p->cell));
  } else {
    if ((st = grow(h, &h->state, &h->state_cap, (size_t)need_state, p, "state scratch")) != RK_OK) return st;
    state = h->state;
  }

  // 1. input projection of every step and direction: a launch of its own, or
  // computed by the blocks the tensor-core recurrence leaves idle
  rk::ProjParams pp{};
  pp.M = (int)(p->seq * p->batch);
  pp.N = sp.G * sp.H;
  pp.K = (int)p->input;
  pp.D = sp.D;
  pp.X = tptr(ops->X, eb);
  pp.W = tptr(ops->W, eb);
  pp.Xw = xw;
  pp.dtype = p->dtype;
  pp.sms = h->sms;
  CUtensorMap tmA{}, tmB{};
  const FusedProj fz = fused_projection(h, p, pl, pp, sp.T > 0 && need_xw > 0, &tmA, &tmB);
  if (sp.T > 0 && need_xw > 0 && !fz.on) {
    if (h->profiling) cudaEventRecord(h->ev[0], stream);
    const bool tc = !(h->flags & RK_FORCE_SIMT_PROJECTION) && rk::projection_tc_supported(pp);
    cudaError_t e = tc ? rk::launch_projection_tc(pp, h->status, h->timeout_ns, stream)
                       : rk::launch_projection_simt(pp, stream);
    if (e != cudaSuccess) return cuda_fail(h, p, "projection launch", e);
    if (h->profiling) cudaEventRecord(h->ev[1], stream);
    h->ev_proj = h->profiling;
    h->launches += 1;
  } else {
    h->ev_proj = false;
  }

  // 2-4. state setup, steps and outputs in one persistent launch
  sp.R = tptr(ops->R, eb);
  sp.Bias = tptr(ops->B, eb);
  sp.lens = static_cast<const int*>(tptr(ops->sequence_lens, 4));
  sp.h0 = tptr(ops->initial_h, eb);
  sp.c0 = tptr(ops->initial_c, eb);
  sp.P = tptr(ops->P, eb);
  sp.Y = tptr_mut(ops->Y, eb);
  sp.Yh = tptr_mut(ops->Y_h, eb);
  sp.Yc = tptr_mut(ops->Y_c, eb);
  sp.xw = xw;
  assign_state(sp, pl, state);
  sp.status = h->status;
  sp.timeout_ns = h->timeout_ns;
  if (pl.kind == rk::kStepGrid || pl.kind == rk::kStepTensor) {
    cudaError_t e = cudaMemsetAsync(state, 0, (size_t)zeroed_state_floats(pl, sp.D) * sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(h, p, "barrier reset", e);
  }
  if (step_wait != nullptr) {
    cudaError_t e = cudaStreamWaitEvent(stream, step_wait, 0);
    if (e != cudaSuccess) return cuda_fail(h, p, "wait for the operand copies", e);
  }
  if (h->profiling) cudaEventRecord(h->ev[2], stream);
  cudaError_t e;
  if (fz.on) {
    StepPlan fp = pl;
    fp.grid = pl.grid + fz.np;
    fp.smem = std::max(pl.smem, rk::projection_tc_smem());
    sp.fused = 1;
    sp.step_ctas = pl.grid;
    sp.pj_M = pp.M;
    sp.pj_K = pp.K;
    sp.pj_vec = (reinterpret_cast<uintptr_t>(xw) % 16 == 0) && (pp.N % 4 == 0);
    sp.xw_groups = fz.groups;
    sp.xw_mpg = fz.mpg;
    sp.xw_ready = sp.counters + fz.counter0;
    // Xw through a ring of 128-row tiles that stays in L2 (used on the
    // device when every row has the same length; else the whole scratch)
    // (a step waits for its whole readiness group of fz.mpg tiles, which
    // must fit the ring next to the tiles still being read)
    const int mt = (pp.M + 127) / 128;
    sp.xw_ring = (mt > 2 * rk::kXwRingTiles && fz.mpg <= rk::kXwRingTiles) ? rk::kXwRingTiles : 0;
    sp.xw_consumers = sp.D > 0 ? pl.grid / sp.D * 8 : 0;
    sp.xw_done = sp.counters + (rk::kStateHeader - sp.D);
    e = rk::step_tc_entry(sp, fp, stream, nullptr, sp.rhglob, &tmA, &tmB);
  } else {
    e = step_dispatch(p->cell, sp, pl, stream, nullptr);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (e == cudaErrorCooperativeLaunchTooLarge)
      return fail(h, RK_ERR_UNSUPPORTED, "%s: step kernel cannot be resident: %s", cell_name(p->cell),
                  cudaGetErrorName(e));
    return cuda_fail(h, p, "step kernel launch", e);
  }
  if (h->profiling) cudaEventRecord(h->ev[3], stream);
  h->ev_step = h->profiling;
  h->launches += 1;
  return RK_OK;
}

}  // namespace

rk_status rk_encode(rk_handle* h, const rk_problem* p, const rk_operands* ops, const rk_scratch* scratch,
                    void* stream_ptr) {
  if (h == nullptr) return RK_ERR_ARG;
  h->last_error.clear();
  rk_status st = validate_all(h, p, ops);
  if (st != RK_OK) return st;
  if (p->batch == 0 || p->hidden == 0) return RK_OK;  // nothing is recorded
  if ((st = ensure_device(h)) != RK_OK) return st;
  return encode_validated(h, p, ops, scratch, static_cast<cudaStream_t>(stream_ptr), nullptr);
}

// The layer with its scratch in the library's fixed device array instead of
// memory from cudaMalloc, for callers that cannot allocate (see rk.h).
rk_status rk_encode_noalloc(rk_handle* h, const rk_problem* p, const rk_operands* ops, void* stream_ptr) {
  if (h == nullptr) return RK_ERR_ARG;
  h->last_error.clear();
  rk_status st = validate_all(h, p, ops);
  if (st != RK_OK) return st;
  if (p->batch == 0 || p->hidden == 0) return RK_OK;  // nothing is recorded
  const int64_t need_state = round_up(state_len(p), 64), need_xw = xw_len(p);
  if (need_state + need_xw > rk::kNoAllocScratchFloats)
    return fail(h, RK_ERR_UNSUPPORTED,
                "%s: no-alloc scratch holds %lld floats (16 MiB); this layer needs %lld (state %lld + xw %lld)",
                cell_name(p->cell), (long long)rk::kNoAllocScratchFloats, (long long)(need_state + need_xw),
                (long long)need_state, (long long)need_xw);
  float* scratch = nullptr;
  int* status = nullptr;
  cudaError_t e = rk::noalloc_scratch(&scratch, &status);
  if (e != cudaSuccess) return cuda_fail(h, p, "no-alloc scratch set-up", e);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int eb = p->dtype == RK_F32 ? 4 : 2;
  // planning needs the device's SM count and shared-memory limit, not a status word
  rk_handle plan_h;
  plan_h.flags = h->flags;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&plan_h.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&plan_h.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(h, p, "device query", e);
  plan_h.device = dev;
  std::copy(std::begin(h->plans), std::end(h->plans), std::begin(plan_h.plans));
  plan_h.plan_next = h->plan_next;
  StepParams sp;
  fill_params_problem(p, &sp);
  StepPlan pl{};
  st = plan_step(&plan_h, p, &sp, &pl, true);
  std::copy(std::begin(plan_h.plans), std::end(plan_h.plans), std::begin(h->plans));
  h->plan_next = plan_h.plan_next;
  if (st != RK_OK) {
    h->last_error = plan_h.last_error;
    return st;
  }
  float* state = scratch;            // 256-byte aligned start of the array
  float* xw = scratch + need_state;  // after the state region
  // the array keeps the previous call's contents: the barrier counters and
  // the status word must start at zero, before either kernel can touch them
  // (the tensor-core projection also reports a wait that gave up there)
  e = cudaMemsetAsync(state, 0, (size_t)zeroed_state_floats(pl, sp.D) * sizeof(float), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int), stream);
  if (e != cudaSuccess) return cuda_fail(h, p, "scratch reset", e);
  h->noalloc_status = status;
  h->ev_proj = h->ev_step = false;
  if (sp.T > 0 && need_xw > 0) {
    rk::ProjParams pp{};
    pp.M = (int)(p->seq * p->batch);
    pp.N = sp.G * sp.H;
    pp.K = (int)p->input;
    pp.D = sp.D;
    pp.X = tptr(ops->X, eb);
    pp.W = tptr(ops->W, eb);
    pp.Xw = xw;
    pp.dtype = p->dtype;
    pp.sms = plan_h.sms;
    if (h->profiling) cudaEventRecord(h->ev[0], stream);
    const bool tc = !(h->flags & RK_FORCE_SIMT_PROJECTION) && rk::projection_tc_supported(pp);
    e = tc ? rk::launch_projection_tc(pp, status, h->timeout_ns, stream) : rk::launch_projection_simt(pp, stream);
    if (e != cudaSuccess) return cuda_fail(h, p, "projection launch", e);
    if (h->profiling) cudaEventRecord(h->ev[1], stream);
    h->ev_proj = h->profiling;
    h->launches += 1;
  }
  sp.R = tptr(ops->R, eb);
  sp.Bias = tptr(ops->B, eb);
  sp.lens = static_cast<const int*>(tptr(ops->sequence_lens, 4));
  sp.h0 = tptr(ops->initial_h, eb);
  sp.c0 = tptr(ops->initial_c, eb);
  sp.P = tptr(ops->P, eb);
  sp.Y = tptr_mut(ops->Y, eb);
  sp.Yh = tptr_mut(ops->Y_h, eb);
  sp.Yc = tptr_mut(ops->Y_c, eb);
  sp.xw = xw;
  assign_state(sp, pl, state);
  sp.status = status;
  sp.timeout_ns = h->timeout_ns;
  if (h->profiling) cudaEventRecord(h->ev[2], stream);
  e = step_dispatch(p->cell, sp, pl, stream, nullptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(h, p, "step kernel launch", e);
  }
  if (h->profiling) cudaEventRecord(h->ev[3], stream);
  h->ev_step = h->profiling;
  h->launches += 1;
  return RK_OK;
}

rk_status rk_set_profiling(rk_handle* h, int32_t enabled) {
  if (h == nullptr) return RK_ERR_ARG;
  if (enabled) {
    rk_status st = ensure_device(h);
    if (st != RK_OK) return st;
    for (auto& ev : h->ev) {
      if (ev == nullptr) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return fail(h, RK_ERR_CUDA, "recurrent: event create: %s", cudaGetErrorName(e));
      }
    }
  }
  h->profiling = enabled != 0;
  h->ev_proj = h->ev_step = false;
  return RK_OK;
}

rk_status rk_last_timings(rk_handle* h, float* projection_ms, float* step_ms) {
  if (h == nullptr || projection_ms == nullptr || step_ms == nullptr) return RK_ERR_ARG;
  *projection_ms = -1.0f;
  *step_ms = -1.0f;
  cudaError_t e = cudaSuccess;
  if (h->ev_proj) {
    e = cudaEventSynchronize(h->ev[1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(projection_ms, h->ev[0], h->ev[1]);
  }
  if (e == cudaSuccess && h->ev_step) {
    e = cudaEventSynchronize(h->ev[3]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(step_ms, h->ev[2], h->ev[3]);
  }
  if (e != cudaSuccess) return fail(h, RK_ERR_CUDA, "recurrent: timings: %s", cudaGetErrorName(e));
  return RK_OK;
}

rk_status rk_encode_host(rk_handle* h, const rk_problem* p, const rk_operands* host_ops, void* stream_ptr) {
  if (h == nullptr) return RK_ERR_ARG;
  h->last_error.clear();
  rk_status st = validate_all(h, p, host_ops);
  if (st != RK_OK) return st;
  if (p->batch == 0 || p->hidden == 0) return RK_OK;
  if ((st = ensure_device(h)) != RK_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int eb = p->dtype == RK_F32 ? 4 : 2;
  Extents ex;
  extents_of(p, &ex);
  struct Item {
    const rk_tensor* src;
    rk_tensor* dst;
    int64_t bytes;
    bool input;
    bool direct_ok;  // read or written by the kernels with plain loads and stores only
  };
  rk_operands dev = {};
  // X and W feed the projection, which reads them with asynchronous copies
  // (cp.async, TMA): always copied to device memory
  Item items[11] = {
      {&host_ops->X, &dev.X, ex.X * eb, true, false},
      {&host_ops->W, &dev.W, ex.W * eb, true, false},
      {&host_ops->R, &dev.R, ex.R * eb, true, true},
      {&host_ops->B, &dev.B, ex.B * eb, true, true},
      {&host_ops->sequence_lens, &dev.sequence_lens, ex.lens * 4, true, true},
      {&host_ops->initial_h, &dev.initial_h, ex.state * eb, true, true},
      {&host_ops->initial_c, &dev.initial_c, ex.state * eb, true, true},
      {&host_ops->P, &dev.P, ex.P * eb, true, true},
      {&host_ops->Y, &dev.Y, ex.Y * eb, false, true},
      {&host_ops->Y_h, &dev.Y_h, ex.state * eb, false, true},
      {&host_ops->Y_c, &dev.Y_c, ex.state * eb, false, true},
  };
  // Page-locked host memory is mapped into the device's address space, so
  // the step kernel reads R, B, the lengths, the initial states and P and
  // writes Y, Y_h, Y_c there directly (over the CPU-GPU link, each byte once)
  // instead of through a copy: a copy costs several microseconds of fixed
  // latency before the first byte moves, which is more than a small layer's
  // whole transfer.  Other host memory is copied.
  void* direct[11] = {};
  if (h->can_map_host) {
    for (int i = 2; i < 11; ++i) {
      const rk_tensor& t = *items[i].src;
      if (!items[i].direct_ok || !t.ptr || items[i].bytes == 0) continue;
      const int elem = (i == 4) ? 4 : eb;
      const char* hp = static_cast<const char*>(t.ptr) + t.offset * elem;
      cudaPointerAttributes a{};
      if (cudaPointerGetAttributes(&a, hp) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) direct[i] = a.devicePointer;
    }
  }
  size_t total = 0;
  size_t offs[11];
  for (int i = 0; i < 11; ++i) {
    offs[i] = total;
    if (items[i].src->ptr && !direct[i]) total += (size_t)round_up(std::max<int64_t>(items[i].bytes, 1), 256);
  }
  if (h->host_arena_cap < total) {
    if (h->host_arena) {
      cudaDeviceSynchronize();
      cudaFree(h->host_arena);
      h->host_arena = nullptr;
      h->host_arena_cap = 0;
    }
    cudaError_t e = cudaMalloc(&h->host_arena, total);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(h, RK_ERR_OOM, "%s: cannot allocate %zu bytes for host operands", cell_name(p->cell), total);
    }
    h->host_arena_cap = total;
  }
  if (h->copy_stream == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&h->copy_ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(h, p, "copy stream set-up", e);
  }
  // W on the caller's stream; X first on the copy stream (forked after the
  // caller's earlier work, joined before the projection), so the two copies
  // overlap; then the other copied operands, joined just before the step
  // kernel, so they land while the projection runs
  cudaError_t e = cudaEventRecord(h->copy_ev[0], stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_stream, h->copy_ev[0], 0);
  if (e != cudaSuccess) return cuda_fail(h, p, "copy stream fork", e);
  for (int i = 0; i < 8; ++i) {
    if (!items[i].src->ptr) continue;
    const int elem = (i == 4) ? 4 : eb;
    items[i].dst->offset = 0;
    items[i].dst->length = items[i].bytes / elem;
    if (direct[i]) {
      items[i].dst->ptr = direct[i];
      continue;
    }
    items[i].dst->ptr = h->host_arena + offs[i];
    if (items[i].bytes > 0) {
      const char* src = static_cast<const char*>(items[i].src->ptr) + items[i].src->offset * elem;
      e = cudaMemcpyAsync(items[i].dst->ptr, src, (size_t)items[i].bytes, cudaMemcpyHostToDevice,
                          i == 1 ? stream : h->copy_stream);
      if (e != cudaSuccess) break;
    }
    if (i == 0 && e == cudaSuccess) e = cudaEventRecord(h->copy_ev[2], h->copy_stream);  // X landed
  }
  for (int i = 8; i < 11; ++i) {
    if (!items[i].src->ptr) continue;
    items[i].dst->offset = 0;
    items[i].dst->length = items[i].bytes / eb;
    items[i].dst->ptr = direct[i] ? direct[i] : h->host_arena + offs[i];
  }
  // on an error past this point the copies already issued are waited for,
  // so that the caller may reuse its host buffers at once
  auto drain = [&]() {
    if (cudaStreamWaitEvent(stream, h->copy_ev[1], 0) != cudaSuccess) cudaStreamSynchronize(h->copy_stream);
    cudaStreamSynchronize(stream);
  };
  cudaError_t j = cudaEventRecord(h->copy_ev[1], h->copy_stream);
  if (e != cudaSuccess || j != cudaSuccess) {
    if (j != cudaSuccess) cudaStreamSynchronize(h->copy_stream);
    else drain();
    return cuda_fail(h, p, "host-to-device copy", e != cudaSuccess ? e : j);
  }
  st = validate_all(h, p, &dev);
  if (st == RK_OK && host_ops->X.ptr) {
    e = cudaStreamWaitEvent(stream, h->copy_ev[2], 0);
    if (e != cudaSuccess) {
      drain();
      return cuda_fail(h, p, "wait for the copy of X", e);
    }
  }
  if (st == RK_OK) st = encode_validated(h, p, &dev, nullptr, stream, h->copy_ev[1]);
  if (st != RK_OK) {
    drain();
    return st;
  }
  for (int i = 8; i < 11; ++i) {
    if (!items[i].src->ptr || items[i].bytes == 0 || direct[i]) continue;
    char* dstp = static_cast<char*>(items[i].src->ptr) + items[i].src->offset * eb;
    e = cudaMemcpyAsync(dstp, items[i].dst->ptr, (size_t)items[i].bytes, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) {
      cudaStreamSynchronize(stream);
      return cuda_fail(h, p, "device-to-host copy", e);
    }
  }
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(h, p, "stream synchronize", e);
  return RK_OK;
}

rk_status rk_status_poll(rk_handle* h, void* stream_ptr) {
  if (h == nullptr) return RK_ERR_ARG;
  if (!h->dev_ready && h->noalloc_status == nullptr) return RK_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int v = 0, w = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && h->dev_ready) e = cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h->dev_ready) e = cudaMemset(h->status, 0, sizeof(int));
  // the fixed array of rk_encode_noalloc has a status word of its own
  if (e == cudaSuccess && h->noalloc_status != nullptr)
    e = cudaMemcpy(&w, h->noalloc_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h->noalloc_status != nullptr) e = cudaMemset(h->noalloc_status, 0, sizeof(int));
  v |= w;
  if (e != cudaSuccess) {
    h->last_error = std::string("recurrent: status poll: ") + cudaGetErrorName(e);
    return RK_ERR_CUDA;
  }
  if (v & 3) {
    h->last_error = "recurrent: a bounded device wait timed out";
    return RK_ERR_TIMEOUT;
  }
  return RK_OK;
}

rk_status rk_set_wait_limit(rk_handle* h, int64_t limit) {
  if (h == nullptr || limit < 1) return RK_ERR_ARG;
  h->timeout_ns = limit;
  return RK_OK;
}

rk_status rk_selftest_timeout(rk_handle* h, void* stream_ptr, int64_t timeout_ns) {
  if (h == nullptr || timeout_ns < 1) return RK_ERR_ARG;
  rk_status st = ensure_device(h);
  if (st != RK_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  rk_problem dummy = {};
  if ((st = grow(h, &h->state, &h->state_cap, rk::kStateHeader, &dummy, "state scratch")) != RK_OK) return st;
  cudaError_t e = cudaMemsetAsync(h->state, 0, sizeof(unsigned), stream);
  if (e == cudaSuccess) e = rk::launch_selftest_timeout(reinterpret_cast<unsigned*>(h->state), h->status, timeout_ns, stream);
  if (e != cudaSuccess) return fail(h, RK_ERR_CUDA, "recurrent: self-test launch: %s", cudaGetErrorName(e));
  h->launches += 1;
  return RK_OK;
}

const char* rk_last_error(const rk_handle* h) { return h ? h->last_error.c_str() : "null handle"; }

uint64_t rk_launch_count(const rk_handle* h) { return h ? h->launches : 0; }

}  // extern "C"
