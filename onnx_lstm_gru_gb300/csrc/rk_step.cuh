// rk_step.cuh -- the persistent recurrent-step kernel (all steps of a layer in
// one launch) for sm_103a.
//
// What it computes follows the web page "Recurrent layers" (onegpu docs):
//   section "How a layer runs", steps 2-4 (state setup, the steps, the
//   outputs) and section "Arithmetic and determinism": per gate row,
//   pre = ((xw + rec) + Wb) + Rb with rec = R . h_prev; then the peephole
//   terms (i, f with the previous c, o with the new c), clip, activation,
//   c = f*c + i*c~, h = o*h_act(c); GRU h = (1 - z)*h~ + z*h_prev, and for
//   linear_before_reset = 0 the candidate's product takes r (.) h_prev of
//   every unit, which needs a second exchange inside the step (step 3 of
//   "How a layer runs").  Section "Semantics": rows whose sequence ended copy
//   their state through, Y is zero past the length, a row of length 0 ends
//   with zero state, Seq = 0 returns the initial state.
//
// How it runs (a GB300 design, not the pages' one-dispatch-per-step design):
//   - The layer is split into independent teams, one per (direction, group
//     of batch rows).  A team owns the whole hidden state of its rows.
//   - Inside a team every CTA owns J hidden units and keeps their G*J rows of
//     R resident in shared memory for the whole layer.
//   - Per step each warp forms RPW row sums for NBC batch rows: lanes take k
//     in float4 slices (k = 4*(32*chunk + lane) + e), each lane chains its
//     terms in increasing k with fused multiply-adds, and the 32 lane sums
//     are combined by a fixed shuffle tree that also transposes the RPW*NBC
//     values across lanes.  The order depends only on the shape, so two runs
//     give the same bits.
//   - One thread per (unit, batch row) does the gate arithmetic.
//   - kStepCluster: a team is a thread-block cluster (up to 16 CTAs); each
//     CTA pushes its new h slice into every peer's shared memory with
//     st.async and the peer's mbarrier counts the bytes, so a step needs no
//     cluster-wide barrier, only that CTA's wait for its own buffer.
//   - kStepGrid: a team spans up to all SMs (cooperative launch); the new h
//     goes to a double-buffered global array (L2 resident) and a counter
//     barrier with a bounded, timed wait orders the steps.
// Every wait is bounded by a deadline on %globaltimer; a wait that runs out
// sets bit 0 of the status word and the kernel winds down without hanging.
#pragma once

#include <cstdint>

#include "rk_elem.cuh"
#include "rk_internal.h"

namespace rk {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
      "r"(__float_as_uint(v.w)), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(bar)
               : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until the grids this one depends on (programmatic dependent launch)
// have completed and their writes are visible; returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel on the stream, if launched as a programmatic
// dependent, start being scheduled.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait for an mbarrier phase with a deadline.  Returns false on timeout.
// One contiguous global -> shared copy on the async proxy (16-byte aligned
// addresses, size a multiple of 16), counted on mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && (long long)(global_ns() - t0) > timeout_ns) return false;
  }
}

// ------------------------------------------------------------------ element access
template <typename T>
__device__ __forceinline__ float load_elem(const T* p) { return Elem<T>::to_f(*p); }

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v) { *p = Elem<T>::from_f(v); }

// 4 consecutive R elements from shared memory as floats (16-byte aligned rows).
template <typename T>
__device__ __forceinline__ float4 load4_smem(const T* p) { return load4_16(p); }
template <>
__device__ __forceinline__ float4 load4_smem<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// ------------------------------------------------------------------ activations
// sigmoid(x) = 1 / (1 + e^-x) and tanh(x) = 1 - 2 / (e^(2x) + 1), written from
// these identities over the __expf intrinsic and the __fdividef fast
// division.  In float32 both stay within about 1e-6 of the exact value
// (__expf is within a few ulp for the arguments that matter, and the forms
// saturate to 0 / +-1 where the exponential overflows); the parity tests hold
// them to the oracle.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float tanh_fast(float x) { return 1.0f - __fdividef(2.0f, __expf(2.0f * x) + 1.0f); }

// The eleven ONNX activations (the pages name them; formulas from the ONNX
// operator definitions).  Comparisons are written so that NaN passes through.
__device__ __forceinline__ float act_eval(int kind, float a, float b, float x) {
  switch (kind) {
    case 0: return sigmoid_fast(x);
    case 1: return tanh_fast(x);
    case 2: return x > 0.0f ? x : (x <= 0.0f ? 0.0f : x);
    case 3: return a * x + b;
    case 4: return x >= 0.0f ? x : (x < 0.0f ? a * x : x);
    case 5: return x > a ? x : (x <= a ? 0.0f : x);
    case 6: return a * tanh_fast(b * x);
    case 7: {
      const float y = a * x + b;
      return y < 0.0f ? 0.0f : (y > 1.0f ? 1.0f : y);
    }
    case 8: return x >= 0.0f ? x : (x < 0.0f ? a * expm1f(x) : x);
    case 9: return x / (1.0f + fabsf(x));
    case 10: return x > 20.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
    default: return __int_as_float(0x7fffffff);
  }
}

// Slot `slot` of direction d.  GEN = false compiles in the ONNX defaults.
template <bool GEN, int DEFAULT_KIND>
__device__ __forceinline__ float act(const StepParams& p, int idx, float x) {
  if constexpr (GEN) {
    return act_eval(p.acts[idx].kind, p.acts[idx].alpha, p.acts[idx].beta, x);
  } else {
    return act_eval(DEFAULT_KIND, 0.0f, 0.0f, x);
  }
}

__device__ __forceinline__ float clip_pre(float c, float x) {
  if (c > 0.0f) {
    if (x > c) return c;
    if (x < -c) return -c;
  }
  return x;
}

// ------------------------------------------------------------------ indexing
__device__ __forceinline__ size_t y_index(const StepParams& p, int t, int d, int b, int j) {
  return p.layout == 0 ? (((size_t)t * p.D + d) * p.N + b) * p.H + j
                       : (((size_t)b * p.S + t) * p.D + d) * p.H + j;
}
__device__ __forceinline__ size_t state_index(const StepParams& p, int d, int b, int j) {
  return p.layout == 0 ? ((size_t)d * p.N + b) * p.H + j : ((size_t)b * p.D + d) * p.H + j;
}
__device__ __forceinline__ size_t xw_index(const StepParams& p, int d, int t, int b, int g, int j) {
  const size_t m = p.layout == 0 ? (size_t)t * p.N + b : (size_t)b * p.S + t;
  return (((size_t)d * p.S * p.N + m) * p.G + g) * p.H + j;
}

// ------------------------------------------------------------------ shuffle tree
// Combine N per-lane partial sums across the 32 lanes of a warp.  At each
// level the lanes whose bit is set keep the upper half of the values and the
// others the lower half, so after the levels lane L holds the full sum of
// value index xreduce_index<N>(L) (duplicated across the lanes that differ
// only in bits below 32/N).  Fixed order: deterministic.
template <int N, int O>
__device__ __forceinline__ void xreduce(float* v, int lane) {
  if constexpr (N > 1) {
    constexpr int H2 = N / 2;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < H2; ++i) {
      const float send = up ? v[i] : v[i + H2];
      const float keep = up ? v[i + H2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
    if constexpr (O > 1) xreduce<H2, O / 2>(v, lane);
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
    if constexpr (O > 1) xreduce<1, O / 2>(v, lane);
  }
}
template <int N>
__device__ __forceinline__ int xreduce_index(int lane) {
  int idx = 0, n = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      n >>= 1;
      if (lane & o) idx += n;
    }
  }
  return idx;
}

// Row sums gs[(row0 + r) * gs_ld + col0 + b] = sum_k Rs[row0 + r][k] * hsrc[b][k]
// for rows [row0, row0 + nrows) (nrows a multiple of RPW) and NBC batch rows.
template <int RPW, int NBC, typename T>
__device__ __forceinline__ void matvec(const T* __restrict__ Rs, int KP, int row0, int nrows,
                                       const float* __restrict__ hsrc, float* __restrict__ gs, int gs_ld,
                                       int col0, int warp, int nwarps, int lane) {
  constexpr int NV = RPW * NBC;
  static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "RPW*NBC must be a power of two <= 32");
  const int nchunks = KP / kKChunk;
  for (int rg = warp; rg * RPW < nrows; rg += nwarps) {
    const int rbase = row0 + rg * RPW;
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.0f;
    for (int kc = 0; kc < nchunks; ++kc) {
      const int k = (kc * 32 + lane) * 4;
      float4 hv[NBC];
#pragma unroll
      for (int b = 0; b < NBC; ++b) hv[b] = *reinterpret_cast<const float4*>(hsrc + (size_t)b * KP + k);
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float4 rv = load4_smem<T>(Rs + (size_t)(rbase + r) * KP + k);
#pragma unroll
        for (int b = 0; b < NBC; ++b) {
          float a = acc[r * NBC + b];
          a = fmaf(rv.x, hv[b].x, a);
          a = fmaf(rv.y, hv[b].y, a);
          a = fmaf(rv.z, hv[b].z, a);
          a = fmaf(rv.w, hv[b].w, a);
          acc[r * NBC + b] = a;
        }
      }
    }
    xreduce<NV, 16>(acc, lane);
    constexpr int DUP = 32 / NV;
    if ((lane & (DUP - 1)) == 0) {
      const int idx = xreduce_index<NV>(lane);
      gs[(size_t)(rbase + idx / NBC) * gs_ld + col0 + (idx % NBC)] = acc[0];
    }
  }
}

// ------------------------------------------------------------------ the kernel
template <int CELL>
struct CellInfo;
template <>
struct CellInfo<0> {  // LSTM: gates i, o, f, c; activations f, g, h
  static constexpr int G = 4, A = 3;
};
template <>
struct CellInfo<1> {  // GRU: gates z, r, h; activations f, g
  static constexpr int G = 3, A = 2;
};
template <>
struct CellInfo<2> {  // RNN: one gate; activation f
  static constexpr int G = 1, A = 1;
};

// Shared-memory layout of one CTA (all offsets in bytes, 16-byte aligned).
struct SmemLayout {
  size_t Rs, hs, rhs, gs, hown, cs, zs, stage, rstage, wb, rb, pp, lens, bar, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline SmemLayout smem_layout(const StepParams& p, int rows_pad, int nbc, int nb, bool grid,
                                                  int elem_bytes) {
  SmemLayout L{};
  const bool lbr0 = p.cell == 1 && !p.lbr;
  const int Jp = rows_pad / p.G;
  size_t o = 0;
  L.Rs = o;   o = align16(o + (size_t)rows_pad * p.KP * elem_bytes);
  // cluster: two full h buffers (and two r.h buffers); grid: one staging chunk
  L.hs = o;   o = align16(o + (size_t)(grid ? 1 : 2) * nbc * p.KP * 4);
  L.rhs = o;  o = align16(o + (size_t)((lbr0 && !grid) ? 2 : 0) * nbc * p.KP * 4);
  L.gs = o;   o = align16(o + (size_t)rows_pad * nb * 4);
  L.hown = o; o = align16(o + (size_t)nb * p.J * 4);
  L.cs = o;   o = align16(o + (size_t)nb * p.J * 4);
  L.zs = o;   o = align16(o + (size_t)(lbr0 ? nb * p.J : 0) * 4);
  L.stage = o;  o = align16(o + (size_t)(grid ? 0 : nb * p.J) * 4);
  L.rstage = o; o = align16(o + (size_t)((lbr0 && !grid) ? nb * p.J : 0) * 4);
  L.wb = o;   o = align16(o + (size_t)p.G * Jp * 4);
  L.rb = o;   o = align16(o + (size_t)p.G * Jp * 4);
  L.pp = o;   o = align16(o + (size_t)3 * Jp * 4);
  L.lens = o; o = align16(o + (size_t)nb * 4);
  L.bar = o;  o = align16(o + 4 * 8);
  L.total = o;
  return L;
}

// Bounded barrier of one team of the grid kernel.  Counter `ctr` only grows;
// the n-th barrier of the launch waits for team_ctas * n arrivals.
__device__ __forceinline__ bool team_barrier(unsigned* ctr, unsigned target, long long timeout_ns, int* status,
                                             int* flag_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    // arrive with release semantics (the CTA's writes, ordered before this
    // thread by the __syncthreads above, are covered); poll with acquire
    // loads, which order every later read -- a full fence before a relaxed
    // add and another after the poll cost 5 % more per step on the reverse
    // LSTM 200 x 4 x 1024 layer
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
    int ok = 1;
    if (ld_acquire_gpu(ctr) < target) {
      const unsigned long long t0 = global_ns();
      for (unsigned it = 1; ld_acquire_gpu(ctr) < target; ++it) {
        if ((it & 31u) == 0 && (long long)(global_ns() - t0) > timeout_ns) {
          atomicOr(status, 1);
          ok = 0;
          break;
        }
      }
    }
    *flag_smem = ok;
  }
  __syncthreads();
  return *flag_smem != 0;
}

// Threads per CTA the kernel is compiled for (registers are budgeted for it).
template <int RPW, int NBC>
struct MaxThreads {
  static constexpr int value = (RPW * NBC >= 32) ? 768 : 512;
};

template <int CELL, typename T, bool GEN, int RPW, int NBC, bool GRID>
__global__ void __launch_bounds__(MaxThreads<RPW, NBC>::value, 1) step_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NT = blockDim.x, nwarps = NT >> 5;
  const int C = p.team_ctas;
  const int rank = GRID ? (int)(blockIdx.x % C) : (int)cluster_ctarank();
  const int team = blockIdx.x / C;
  const int d = team / p.teams_per_dir;
  const int b0 = (team % p.teams_per_dir) * p.nb;
  const int nbt = min(p.nb, p.N - b0);
  const int J = p.J, KP = p.KP, H = p.H;
  const int Jp = p.rows_pad / G;
  const int j0 = rank * J;
  const int Jc = max(0, min(J, H - j0));
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const bool lbr0 = (CELL == 1) && !p.lbr;
  // row stride of gs: the team's batch rows rounded up to whole chunks
  const int nb_ld = GRID ? ((p.nb + NBC - 1) / NBC) * NBC : NBC;
  const bool has_p = CELL == 0 && p.P != nullptr;

  const SmemLayout L = smem_layout(p, p.rows_pad, NBC, nb_ld, GRID, (int)sizeof(T));
  T* Rs = reinterpret_cast<T*>(smem + L.Rs);
  float* hs = reinterpret_cast<float*>(smem + L.hs);
  float* rhs = reinterpret_cast<float*>(smem + L.rhs);
  float* gs = reinterpret_cast<float*>(smem + L.gs);
  float* hown = reinterpret_cast<float*>(smem + L.hown);
  float* cs = reinterpret_cast<float*>(smem + L.cs);
  float* zs = reinterpret_cast<float*>(smem + L.zs);
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  float* rstage = reinterpret_cast<float*>(smem + L.rstage);
  float* wb_s = reinterpret_cast<float*>(smem + L.wb);
  float* rb_s = reinterpret_cast<float*>(smem + L.rb);
  float* pp_s = reinterpret_cast<float*>(smem + L.pp);
  int* lens_s = reinterpret_cast<int*>(smem + L.lens);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);  // [0,1] h buffers, [2,3] r.h buffers
  __shared__ int flag_smem;

  const T* R = static_cast<const T*>(p.R);
  const T* Bias = static_cast<const T*>(p.Bias);
  const T* P = static_cast<const T*>(p.P);
  const T* h0 = static_cast<const T*>(p.h0);
  const T* c0 = static_cast<const T*>(p.c0);
  T* Y = static_cast<T*>(p.Y);

  // ---------------- prologue: R slice, biases, peepholes, lengths, state (step 2)
  {
    const size_t GH = (size_t)G * H;
    const int nrow = p.rows_pad;
    for (size_t e = tid; e < (size_t)nrow * KP; e += NT) {
      const int lr = (int)(e / KP), k = (int)(e % KP);
      const int g = lr / Jp, jl = lr % Jp;
      Rs[e] = (g < G && jl < Jc && k < H) ? R[((size_t)d * GH + (size_t)g * H + j0 + jl) * H + k]
                                          : static_cast<T>(0.0f);
    }
    for (int e = tid; e < G * Jp; e += NT) {
      const int g = e / Jp, jl = e % Jp;
      const bool ok = jl < Jc && Bias != nullptr;
      const size_t row = (size_t)g * H + j0 + jl;
      wb_s[e] = ok ? load_elem<T>(Bias + (size_t)d * 2 * GH + row) : 0.0f;
      rb_s[e] = ok ? load_elem<T>(Bias + (size_t)d * 2 * GH + GH + row) : 0.0f;
    }
    for (int e = tid; e < 3 * Jp; e += NT) {
      const int g = e / Jp, jl = e % Jp;
      pp_s[e] = (CELL == 0 && P != nullptr && jl < Jc) ? load_elem<T>(P + (size_t)d * 3 * H + (size_t)g * H + j0 + jl)
                                                       : 0.0f;
    }
    for (int bl = tid; bl < nb_ld; bl += NT) {
      int len = p.T;
      if (bl < nbt && p.lens != nullptr) {
        len = p.lens[b0 + bl];
        len = len < 0 ? 0 : (len > p.S ? p.S : len);
        len = len > p.T ? p.T : len;
      }
      lens_s[bl] = bl < nbt ? len : 0;
    }
    for (int e = tid; e < nbt * J; e += NT) {
      const int bl = e / J, jl = e % J;
      float hv = 0.0f, cv = 0.0f;
      if (jl < Jc) {
        const size_t si = state_index(p, d, b0 + bl, j0 + jl);
        if (h0 != nullptr) hv = load_elem<T>(h0 + si);
        if (CELL == 0 && c0 != nullptr) cv = load_elem<T>(c0 + si);
      }
      hown[e] = hv;
      cs[e] = cv;
    }
    if constexpr (!GRID) {
      // full initial h of the team's rows into buffer 0; zero buffer 1 and the r.h buffers
      for (size_t e = tid; e < (size_t)2 * NBC * KP; e += NT) {
        const int buf = (int)(e / ((size_t)NBC * KP));
        const int bl = (int)((e / KP) % NBC), k = (int)(e % KP);
        float v = 0.0f;
        if (buf == 0 && bl < nbt && k < H && h0 != nullptr) v = load_elem<T>(h0 + state_index(p, d, b0 + bl, k));
        hs[e] = v;
        if (lbr0) rhs[e] = 0.0f;
      }
      if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
        fence_mbar_init_cluster();
      }
      cluster_sync_all();
    } else {
      // publish this CTA's initial h into the global exchange buffer 0
      for (int e = tid; e < nbt * Jc; e += NT) {
        const int bl = e / Jc, jl = e % Jc;
        p.hglob[((size_t)d * p.N + b0 + bl) * KP + j0 + jl] = hown[bl * J + jl];
      }
      // staged rows are copied in whole (H columns each): the columns past
      // H stay zero from here on (the grid kernel stages h and r.h alike in
      // its one chunk buffer hs)
      for (size_t e = tid; e < (size_t)NBC * KP; e += NT) hs[e] = 0.0f;
      if (tid == 0) mbar_init(smem_u32(&bars[0]), 1);  // staged rows landed
      // the exchange buffer is written by ordinary stores and read by bulk copies
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }

  unsigned nbar = 0;  // grid barriers passed so far
  bool alive = true;
  if constexpr (GRID) {
    alive = team_barrier(p.counters + team, (unsigned)C * (++nbar), p.timeout_ns, p.status, &flag_smem);
  }

  // Stage the batch rows [c0, c0 + NBC) of a global exchange buffer (grid
  // kernel): one bulk copy of H floats per row when rows are a whole number
  // of 16 bytes (rows past the team's batch keep stale values whose sums no
  // gate reads), else element loads.
  const bool bulk_rows = (H % 4) == 0;
  uint32_t stage_phase = 0;
  auto load_chunk = [&](const float* src, int c0) -> bool {
    if (bulk_rows) {
      const int nrows = min(NBC, nbt - c0);
      if (tid == 0) {
        // the writers' ordinary stores, acquired by the team barrier, are
        // read by the async proxy; this block's reads of the previous rows
        // come before the async proxy rewrites them
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(smem_u32(&bars[0]), (uint32_t)nrows * (uint32_t)H * 4u);
        for (int bl = 0; bl < nrows; ++bl)
          bulk_copy_g2s(smem_u32(hs + (size_t)bl * KP), src + ((size_t)d * p.N + b0 + c0 + bl) * KP, (uint32_t)H * 4u,
                        smem_u32(&bars[0]));
      }
      const bool ok = mbar_wait_bounded(smem_u32(&bars[0]), stage_phase & 1u, p.timeout_ns);
      ++stage_phase;
      return ok;
    }
    const int nk4 = KP / 4;
    for (int e = tid; e < NBC * nk4; e += NT) {
      const int bl = e / nk4, k = (e % nk4) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c0 + bl < nbt && k < H) {
        const float* q = src + ((size_t)d * p.N + b0 + c0 + bl) * KP + k;
        if (k + 3 < H) {
          v = __ldcg(reinterpret_cast<const float4*>(q));
        } else {
          v.x = __ldcg(q);
          if (k + 1 < H) v.y = __ldcg(q + 1);
          if (k + 2 < H) v.z = __ldcg(q + 2);
        }
      }
      *reinterpret_cast<float4*>(hs + (size_t)bl * KP + k) = v;
    }
    return true;
  };

  // Row sums for rows [row0, row0 + nrows) against the current h (or r.h).
  auto products = [&](int row0, int nrows, const float* cluster_src, const float* global_src) {
    if constexpr (!GRID) {
      matvec<RPW, NBC, T>(Rs, KP, row0, nrows, cluster_src, gs, NBC, 0, warp, nwarps, lane);
    } else {
      for (int c0 = 0; c0 < nbt; c0 += NBC) {
        if (!load_chunk(global_src, c0) && tid == 0) atomicOr(p.status, 1);  // the barriers after it still pass
        __syncthreads();
        matvec<RPW, NBC, T>(Rs, KP, row0, nrows, hs, gs, nb_ld, c0, warp, nwarps, lane);
        __syncthreads();
      }
    }
  };

  // Push this CTA's slice (stage[bl][0..Jc)) into buffer `dst` of every CTA of the cluster.
  auto push_slice = [&](const float* src_stage, float* dst, uint64_t* bar) {
    const uint32_t dst_base = smem_u32(dst);
    const uint32_t bar_local = smem_u32(bar);
    const bool vec = ((J & 3) == 0) && ((H & 3) == 0);
    if (vec) {
      const int per_row = Jc >> 2, per_peer = nbt * per_row, total = C * per_peer;
      for (int i = tid; i < total; i += NT) {
        const int q = i / per_peer, rem = i % per_peer, bl = rem / per_row, v = rem % per_row;
        const float4 val = *reinterpret_cast<const float4*>(src_stage + bl * J + v * 4);
        const uint32_t a = dst_base + (uint32_t)(((size_t)bl * KP + j0 + v * 4) * 4);
        st_async_v4(map_to_rank(a, q), val, map_to_rank(bar_local, q));
      }
    } else {
      const int per_peer = nbt * Jc, total = C * per_peer;
      for (int i = tid; i < total; i += NT) {
        const int q = i / per_peer, rem = i % per_peer, bl = rem / Jc, jl = rem % Jc;
        const uint32_t a = dst_base + (uint32_t)(((size_t)bl * KP + j0 + jl) * 4);
        st_async_b32(map_to_rank(a, q), src_stage[bl * J + jl], map_to_rank(bar_local, q));
      }
    }
  };

  const int npairs = Jc * nbt;
  const uint32_t h_bytes = (uint32_t)nbt * (uint32_t)H * 4u;
  // The cluster kernel's launch may overlap the projection that writes Xw
  // (programmatic dependent launch); wait for it before the first Xw read.
  // Xw is read with coherent loads (__ldcg): a read-only-path load may be
  // scheduled ahead of the wait.
  if constexpr (!GRID) grid_dependency_wait();

  // ---------------- the steps (step 3), all in this launch
  for (int s = 0; s < p.T && alive; ++s) {
    const int cur = s & 1, nxt = cur ^ 1;
    if constexpr (!GRID) {
      if (tid == 0) {
        if (s + 1 < p.T) mbar_arrive_expect_tx(smem_u32(&bars[nxt]), h_bytes);
        if (lbr0) mbar_arrive_expect_tx(smem_u32(&bars[2 + cur]), h_bytes);
      }
    }
    // prefetch this thread's xw (first pair) before waiting on h
    float xwv[G];
    int pj = 0, pb = 0, pL = 0, pt = 0;
    bool pact = false;
    if (tid < npairs) {
      pj = tid % Jc;
      pb = tid / Jc;
      pL = lens_s[pb];
      pact = s < pL;
      pt = pact ? (reverse ? pL - 1 - s : s) : s;
#pragma unroll
      for (int g = 0; g < G; ++g) xwv[g] = pact ? __ldcg(p.xw + xw_index(p, d, pt, b0 + pb, g, j0 + pj)) : 0.0f;
    }
    bool timed_out = false;
    if constexpr (!GRID) {
      if (s >= 1) timed_out = !mbar_wait_bounded(smem_u32(&bars[cur]), (uint32_t)(((s - 1) >> 1) & 1), p.timeout_ns);
    }
    // rec = R . h_prev for all gate rows (GRU lbr=0: z and r rows only)
    products(0, lbr0 ? 2 * Jp : G * Jp, hs + (size_t)cur * NBC * KP, p.hglob + (size_t)cur * p.D * p.N * KP);
    if constexpr (!GRID) {
      if (__syncthreads_or(timed_out)) {
        if (tid == 0) atomicOr(p.status, 1);
        alive = false;
        break;
      }
    }

    if (lbr0) {
      // GRU, linear_before_reset = 0: z, r, then r (.) h_prev of every unit is exchanged
      for (int idx = tid; idx < npairs; idx += NT) {
        const int jl = idx % Jc, bl = idx / Jc;
        const int L = lens_s[bl];
        const bool active = s < L;
        const int t = active ? (reverse ? L - 1 - s : s) : s;
        float xz, xr;
        if (idx == tid) {
          xz = xwv[0];
          xr = xwv[1];
        } else {
          xz = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, 0, j0 + jl)) : 0.0f;
          xr = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, 1, j0 + jl)) : 0.0f;
        }
        const float hp = hown[bl * J + jl];
        const float pz = ((xz + gs[(size_t)(0 * Jp + jl) * nb_ld + bl]) + wb_s[0 * Jp + jl]) + rb_s[0 * Jp + jl];
        const float pr = ((xr + gs[(size_t)(1 * Jp + jl) * nb_ld + bl]) + wb_s[1 * Jp + jl]) + rb_s[1 * Jp + jl];
        const float z = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pz));
        const float r = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pr));
        zs[bl * J + jl] = z;
        const float rh = r * hp;
        if constexpr (GRID) {
          p.rhglob[((size_t)d * p.N + b0 + bl) * KP + j0 + jl] = rh;
        } else {
          rstage[bl * J + jl] = rh;
        }
      }
      if constexpr (GRID) {
        asm volatile("fence.proxy.async.global;" ::: "memory");  // r.h is read by bulk copies
        alive = team_barrier(p.counters + team, (unsigned)C * (++nbar), p.timeout_ns, p.status, &flag_smem);
        if (!alive) break;
      } else {
        __syncthreads();
        push_slice(rstage, rhs + (size_t)cur * NBC * KP, &bars[2 + cur]);
        timed_out = !mbar_wait_bounded(smem_u32(&bars[2 + cur]), (uint32_t)((s >> 1) & 1), p.timeout_ns);
        if (__syncthreads_or(timed_out)) {
          if (tid == 0) atomicOr(p.status, 1);
          alive = false;
          break;
        }
      }
      products(2 * Jp, Jp, rhs + (size_t)cur * NBC * KP, p.rhglob);
      if constexpr (!GRID) __syncthreads();
    }

    // gate arithmetic and state update, one (unit, batch row) pair per thread
    for (int idx = tid; idx < npairs; idx += NT) {
      const int jl = idx % Jc, bl = idx / Jc;
      const int L = lens_s[bl];
      const bool active = s < L;
      const int t = active ? (reverse ? L - 1 - s : s) : s;
      float xv[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (idx == tid) {
          xv[g] = xwv[g];
        } else {
          xv[g] = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, g, j0 + jl)) : 0.0f;
        }
      }
      const float hp = hown[bl * J + jl];
      float hn = hp;
      if (active) {
        float pre[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int lr = g * Jp + jl;
          pre[g] = ((xv[g] + gs[(size_t)lr * nb_ld + bl]) + wb_s[lr]) + rb_s[lr];
        }
        if constexpr (CELL == 0) {
          const float cp = cs[bl * J + jl];
          float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
          if (has_p) {
            pi = pi + pp_s[0 * Jp + jl] * cp;
            pf = pf + pp_s[2 * Jp + jl] * cp;
          }
          const float ig = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pi));
          const float fg = p.input_forget ? 1.0f - ig : act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pf));
          const float cg = act<GEN, 1>(p, d * A + 1, clip_pre(p.clip, pc));
          const float cn = fg * cp + ig * cg;
          if (has_p) po = po + pp_s[1 * Jp + jl] * cn;
          const float og = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, po));
          hn = og * act<GEN, 1>(p, d * A + 2, cn);
          cs[bl * J + jl] = cn;
        } else if constexpr (CELL == 1) {
          float z, ph;
          if (lbr0) {
            z = zs[bl * J + jl];
            ph = pre[2];  // ((xw_h + R_h.(r.h)) + Wb_h) + Rb_h
          } else {
            z = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pre[0]));
            const float r = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pre[1]));
            const int lr = 2 * Jp + jl;
            ph = (xv[2] + r * (gs[(size_t)lr * nb_ld + bl] + rb_s[lr])) + wb_s[lr];
          }
          const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(p.clip, ph));
          hn = (1.0f - z) * hc + z * hp;
        } else {
          hn = act<GEN, 1>(p, d * A + 0, clip_pre(p.clip, pre[0]));
        }
      }
      hown[bl * J + jl] = hn;
      if (Y != nullptr) store_elem<T>(Y + y_index(p, t, d, b0 + bl, j0 + jl), active ? hn : 0.0f);
      if constexpr (GRID) {
        p.hglob[(size_t)nxt * p.D * p.N * KP + ((size_t)d * p.N + b0 + bl) * KP + j0 + jl] = hn;
      } else {
        stage[bl * J + jl] = hn;
      }
    }
    if (s + 1 < p.T) {
      if constexpr (GRID) {
        asm volatile("fence.proxy.async.global;" ::: "memory");  // h is read by bulk copies
        alive = team_barrier(p.counters + team, (unsigned)C * (++nbar), p.timeout_ns, p.status, &flag_smem);
      } else {
        __syncthreads();
        push_slice(stage, hs + (size_t)nxt * NBC * KP, &bars[nxt]);
      }
    }
  }

  // ---------------- outputs (step 4): zero Y past the loop, final states
  __syncthreads();
  if (alive) {
    for (int idx = tid; idx < npairs; idx += NT) {
      const int jl = idx % Jc, bl = idx / Jc;
      if (Y != nullptr)
        for (int t = p.T; t < p.S; ++t) store_elem<T>(Y + y_index(p, t, d, b0 + bl, j0 + jl), 0.0f);
      const bool zero = p.S > 0 && lens_s[bl] == 0;
      const size_t si = state_index(p, d, b0 + bl, j0 + jl);
      if (p.Yh != nullptr) store_elem<T>(static_cast<T*>(p.Yh) + si, zero ? 0.0f : hown[bl * J + jl]);
      if (CELL == 0 && p.Yc != nullptr) store_elem<T>(static_cast<T*>(p.Yc) + si, zero ? 0.0f : cs[bl * J + jl]);
    }
  }
  if constexpr (!GRID) cluster_sync_all();
}

}  // namespace rk
