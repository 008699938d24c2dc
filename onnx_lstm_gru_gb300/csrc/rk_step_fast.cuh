// rk_step_fast.cuh -- latency-first persistent step kernel for layers whose
// team (one thread-block cluster) holds one batch row and whose R rows fit in
// registers.
//
// What it computes is the same as rk_step.cuh (web page "Recurrent layers",
// sections "How a layer runs" and "Arithmetic and determinism"): per step and
// gate row pre = ((xw + rec) + Wb) + Rb with rec = R_row . h_prev, then
// peepholes, clip, activation and state update; a GRU with
// linear_before_reset = 0 exchanges r (.) h_prev of every unit before the
// candidate's product.  xw comes from the projection kernel (Xw scratch).
//
// Layout: one cluster of C CTAs per (direction, batch row); CTA `rank` owns
// hidden units [j0, j0 + J) with J <= 32.  Warp w owns U whole units
// (U = 4 for LSTM and GRU when R's rows are short enough, else 2; 8 for
// RNN): all G*U of their rows of R live in the warp's registers for the whole
// layer (lanes hold k = 4*(32*chunk + lane) + e).  Each exchange message then
// carries 4 units (16 bytes): the cost of an exchange grows with the number
// of st.async messages a CTA receives, so fewer, larger messages matter.
// Per step a warp
//   1. waits on its CTA's mbarrier for h_prev (all H units, pushed by every
//      CTA of the cluster with st.async),
//   2. forms its row sums (each lane chains its terms in increasing k, then a
//      fixed shuffle tree folds the 32 lanes), so runs are bit-identical,
//   3. gathers each unit's gate sums into lane u by shuffles and does the gate
//      arithmetic there (h, c, biases, peepholes and the step's xw,
//      prefetched two steps ahead, all in registers),
//   4. writes Y and pushes its U new h values into every CTA of the cluster.
// No barrier inside a CTA: the only synchronisation is the byte-counting
// mbarrier of each h (and r.h) exchange.  Every wait is bounded by a deadline
// on %globaltimer; a warp whose wait gives up sets the status word, marks the
// CTA aborted and leaves the step loop, and the others follow at their next
// wait.
#pragma once

#include "rk_step_common.cuh"

namespace rk {

// Register rows a warp holds: G * U rounded up to a power of two (8 or 16).
template <int CELL, int U>
struct FastRows {
  static constexpr int G = CELL == 0 ? 4 : (CELL == 1 ? 3 : 1);
  static constexpr int value = (G * U <= 8) ? 8 : 16;
};

struct FastSmem {
  size_t hs, rhs, bar, total;
};

// Shared memory of the fast kernel (offsets in bytes).
__host__ __device__ inline FastSmem fast_smem_layout(const StepParams& p) {
  FastSmem L{};
  size_t o = 0;
  const bool lbr0 = p.cell == 1 && !p.lbr;
  L.hs = o;  o = align16(o + 2 * (size_t)p.KP * 4);
  L.rhs = o; o = align16(o + (lbr0 ? 2 * (size_t)p.KP * 4 : 0));
  L.bar = o; o = align16(o + 4 * 8);
  L.total = o;
  return L;
}

// R fragment kept in registers: 4 consecutive k of one row, in the storage
// type (two packed 16-bit pairs for Half and bfloat16).
template <typename T>
struct RFrag {
  uint2 v;
  __device__ __forceinline__ float4 get() const {
    const float2 a = Elem<T>::pair_to_f(v.x);
    const float2 b = Elem<T>::pair_to_f(v.y);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  // the values come from the stored tensor, so the rounding is exact
  __device__ __forceinline__ void set(const float e[4]) {
    v.x = Elem<T>::pair_from_f(e[0], e[1]);
    v.y = Elem<T>::pair_from_f(e[2], e[3]);
  }
};
// bfloat16: the float32 value of bfloat16 bits b is b << 16, so a packed pair
// unpacks with a shift and a mask.  Written as volatile asm so that the
// compiler keeps the unpacking inside the step loop: hoisted out of it (R is
// loop-invariant) it would hold every fragment twice and spill.
template <>
struct RFrag<__nv_bfloat16> {
  uint2 v;
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    uint32_t lo, hi;
    asm volatile("shl.b32 %0, %1, 16;" : "=r"(lo) : "r"(u));
    asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(hi) : "r"(u));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
  }
  __device__ __forceinline__ float4 get() const {
    const float2 a = unpack(v.x);
    const float2 b = unpack(v.y);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  // the values come from the stored tensor, so the rounding is exact
  __device__ __forceinline__ void set(const float e[4]) {
    v.x = Elem<__nv_bfloat16>::pair_from_f(e[0], e[1]);
    v.y = Elem<__nv_bfloat16>::pair_from_f(e[2], e[3]);
  }
};
template <>
struct RFrag<float> {
  float4 v;
  __device__ __forceinline__ float4 get() const { return v; }
  __device__ __forceinline__ void set(const float e[4]) { v = make_float4(e[0], e[1], e[2], e[3]); }
};

// Fragment of 4 consecutive k of one row of R (elements k0 .. k0 + 3 of
// `row`): one 16-byte (float32) or 8-byte (16-bit) load when the four are
// inside the row and aligned, else element loads with zeros past H.  The
// prologue's R loads are what the step kernel spends before its first step.
template <typename T>
__device__ __forceinline__ void load_frag(RFrag<T>& f, const T* row, int k0, int H, bool ok) {
  const T* src = row + k0;
  if (ok && k0 + 3 < H && (reinterpret_cast<uintptr_t>(src) % (4 * sizeof(T))) == 0) {
    if constexpr (sizeof(T) == 4) f.v = __ldg(reinterpret_cast<const float4*>(src));
    else f.v = __ldg(reinterpret_cast<const uint2*>(src));
    return;
  }
  float e[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) e[q] = (ok && k0 + q < H) ? load_elem<T>(src + q) : 0.0f;
  f.set(e);
}

__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(bar)
               : "memory");
}

// Row sums with a shuffle tree that needs no selects.  Lane l keeps the NR
// rows of a block in the lane-dependent order i -> i ^ perm_mask<NR>(l) (the
// rows' registers are loaded that way), so at every level each lane adds the
// upper half of its partial sums, received from its partner lane, to its lower
// half.  Afterwards lane l holds the full sum of row perm_mask<NR>(l) of the
// block, i.e. row r sits in lanes r * (32 / NR) ... r * (32 / NR) + 32/NR - 1.
template <int NR>
__host__ __device__ constexpr int log2c() { return NR <= 1 ? 0 : 1 + log2c<NR / 2>(); }
template <int NR>
__device__ __forceinline__ int perm_mask(int lane) { return (lane >> (5 - log2c<NR>())) & (NR - 1); }
template <int NR>
__device__ __forceinline__ int row_lane(int r) { return r << (5 - log2c<NR>()); }

template <int N, int O>
__device__ __forceinline__ void fold(float* v) {
  if constexpr (N > 1) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + N / 2], O);
    if constexpr (O > 1) fold<N / 2, O / 2>(v);
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
    if constexpr (O > 1) fold<1, O / 2>(v);
  }
}

// Sums of register rows R0 .. R0+NR-1 (a block stored in permuted order)
// against h (KV float4 slices per lane); each lane chains its terms in
// increasing k, then fold() combines the 32 lanes in a fixed order.
template <int R0, int NR, typename T, int KV, int RW>
__device__ __forceinline__ float rowsums(const RFrag<T> (&R)[RW][KV], const float* __restrict__ h, int lane) {
  float4 hv[KV];
#pragma unroll
  for (int kc = 0; kc < KV; ++kc) hv[kc] = *reinterpret_cast<const float4*>(h + (kc * 32 + lane) * 4);
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float a = 0.0f;
#pragma unroll
    for (int kc = 0; kc < KV; ++kc) {
      const float4 rv = R[R0 + r][kc].get();
      a = fmaf(rv.x, hv[kc].x, a);
      a = fmaf(rv.y, hv[kc].y, a);
      a = fmaf(rv.z, hv[kc].z, a);
      a = fmaf(rv.w, hv[kc].w, a);
    }
    acc[r] = a;
  }
  fold<NR, 16>(acc);
  return acc[0];
}

// Grouped layout (LSTM and RNN): the warp's 32 lanes form 4 groups of 8;
// group g holds rows g * NRG ... g * NRG + NRG - 1 (NRG = RW / 4, a power of
// two) and lane i of a group holds, for each of them, the 4 KV chunks of 4
// consecutive k at k = (c * 8 + i) * 4 + e.  A row's 8 lanes chain their
// terms in increasing k, then fold() combines them over 3 levels (lanes
// xor 4, 2, 1) instead of 5; rows are kept in the order
// rho -> rho ^ group_perm<NRG>(i), so that afterwards lane 8 g + i holds the
// full sum of row g * NRG + group_perm<NRG>(i).
template <int NRG>
__device__ __forceinline__ int group_perm(int lane) { return ((lane & 7) >> (3 - log2c<NRG>())) & (NRG - 1); }
template <int NRG>
__device__ __forceinline__ int group_row_lane(int r) { return 8 * (r / NRG) + ((r % NRG) << (3 - log2c<NRG>())); }

template <int NRG, typename T, int NCH>
__device__ __forceinline__ float rowsums_grouped(const RFrag<T> (&R)[NRG][NCH], const float* __restrict__ h, int lane) {
  const int i = lane & 7;
  float4 hv[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) hv[c] = *reinterpret_cast<const float4*>(h + (c * 8 + i) * 4);
  float acc[NRG];
#pragma unroll
  for (int r = 0; r < NRG; ++r) {
    float a = 0.0f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const float4 rv = R[r][c].get();
      a = fmaf(rv.x, hv[c].x, a);
      a = fmaf(rv.y, hv[c].y, a);
      a = fmaf(rv.z, hv[c].z, a);
      a = fmaf(rv.w, hv[c].w, a);
    }
    acc[r] = a;
  }
  fold<NRG, 4>(acc);
  return acc[0];
}

template <int CELL, int RW>
struct FastGrouped {
  // LSTM and RNN whose rows per group (RW / 4) are a power of two
  static constexpr bool value = CELL != 1 && RW % 4 == 0 && ((RW / 4) & (RW / 4 - 1)) == 0;
};

// PLAIN: no clip, no peepholes, no input_forget (the options compile out).
template <int CELL, typename T, bool GEN, int KV, int U, bool PLAIN>
__global__ void __launch_bounds__(U == 2 ? 512 : 256, 1) step_fast_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  constexpr int RW = FastRows<CELL, U>::value;  // register rows per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = p.team_ctas;
  const int rank = (int)cluster_ctarank();
  const int team = blockIdx.x / C;
  const int d = team / p.N, b = team % p.N;  // one batch row per team
  const int J = p.J, H = p.H, KP = p.KP;
  const int j0 = rank * J;
  const int Jc = max(0, min(J, H - j0));
  const int wu0 = warp * U;                 // first local unit of this warp
  const int Uc = max(0, min(U, Jc - wu0));  // units this warp owns
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const bool lbr0 = (CELL == 1) && !p.lbr;
  const int S = p.S, Tn = p.T;

  const FastSmem L = fast_smem_layout(p);
  float* hs = reinterpret_cast<float*>(smem + L.hs);
  float* rhs = reinterpret_cast<float*>(smem + L.rhs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);  // h[2], r.h[2]
  __shared__ volatile int abort_flag;

  const T* R = static_cast<const T*>(p.R);
  const T* Bias = static_cast<const T*>(p.Bias);
  const T* P = static_cast<const T*>(p.P);
  const T* h0 = static_cast<const T*>(p.h0);
  const T* c0 = static_cast<const T*>(p.c0);
  T* Y = static_cast<T*>(p.Y);
  const size_t GH = (size_t)G * H;

  int len = Tn;
  if (p.lens != nullptr) {
    len = p.lens[b];
    len = len < 0 ? 0 : (len > S ? S : len);
    len = len > Tn ? Tn : len;
  }

  // ---------------- prologue: R rows into registers, h_0, per-unit state
  // register i of this lane holds row row_of(i) of the warp's rows (g * U + u)
  auto row_of = [&](int i) -> int {
    if (lbr0) {
      if (i < 2 * U) return i ^ perm_mask<2 * U>(lane);
      if (i < 3 * U) return 2 * U + ((i - 2 * U) ^ perm_mask<U>(lane));
      return i;
    }
    return i ^ perm_mask<RW>(lane);
  };
  constexpr bool GROUPED = FastGrouped<CELL, RW>::value;
  constexpr int NRG = GROUPED ? RW / 4 : 1;   // rows per 8-lane group
  constexpr int NCH = 4 * KV;                 // 4-k chunks per lane and row (grouped)
  RFrag<T> Rr[GROUPED ? 1 : RW][KV];
  RFrag<T> Rg[NRG][GROUPED ? NCH : 1];
  if constexpr (GROUPED) {
    const int grp = lane >> 3, gi = lane & 7;
#pragma unroll
    for (int rho = 0; rho < NRG; ++rho) {
      const int r = grp * NRG + (rho ^ group_perm<NRG>(lane));
      const int g = r / U, u = r % U;
      const bool ok = g < G && u < Uc;
      const T* row = R + ((size_t)d * GH + (size_t)g * H + j0 + wu0 + u) * H;
#pragma unroll
      for (int c = 0; c < NCH; ++c) load_frag<T>(Rg[rho][c], row, (c * 8 + gi) * 4, H, ok);
    }
  } else {
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int r = row_of(i);
      const int g = r / U, u = r % U;
      const bool ok = g < G && u < Uc;
      const T* row = R + ((size_t)d * GH + (size_t)g * H + j0 + wu0 + u) * H;
#pragma unroll
      for (int kc = 0; kc < KV; ++kc) load_frag<T>(Rr[i][kc], row, (kc * 32 + lane) * 4, H, ok);
    }
  }
  for (int e = tid; e < 2 * KP; e += blockDim.x) {
    const int k = e % KP;
    hs[e] = (e < KP && k < H && h0 != nullptr) ? load_elem<T>(h0 + state_index(p, d, b, k)) : 0.0f;
    if (lbr0) rhs[e] = 0.0f;
  }
  // lane u < Uc of the warp owns unit uj = j0 + wu0 + u
  const bool gl = lane < Uc;
  const int uj = j0 + wu0 + (gl ? lane : 0);
  float hreg = 0.0f, creg = 0.0f, wbv[G], rbv[G], ppv[3];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    wbv[g] = (gl && Bias != nullptr) ? load_elem<T>(Bias + (size_t)d * 2 * GH + (size_t)g * H + uj) : 0.0f;
    rbv[g] = (gl && Bias != nullptr) ? load_elem<T>(Bias + (size_t)d * 2 * GH + GH + (size_t)g * H + uj) : 0.0f;
  }
#pragma unroll
  for (int g = 0; g < 3; ++g)
    ppv[g] = (CELL == 0 && gl && P != nullptr) ? load_elem<T>(P + (size_t)d * 3 * H + (size_t)g * H + uj) : 0.0f;
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;
  if (gl) {
    const size_t si = state_index(p, d, b, uj);
    hreg = h0 != nullptr ? load_elem<T>(h0 + si) : 0.0f;
    creg = (CELL == 0 && c0 != nullptr) ? load_elem<T>(c0 + si) : 0.0f;
  }
  const size_t ystride = p.layout == 0 ? (size_t)p.D * p.N * H : (size_t)p.D * H;
  T* ybase = (Y != nullptr && gl) ? Y + y_index(p, 0, d, b, uj) : nullptr;
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_flag = 0;
    fence_mbar_init_cluster();
  }
  cluster_sync_all();

  // ---------------- the push of this warp's units into every CTA
  // vector form (whole warps, unit offsets aligned to the message size):
  // U = 2 -> one 8-byte st.async per peer (lanes q < C); U = 4 -> one 16-byte
  // st.async per peer; U = 8 -> two 16-byte st.async per peer (lanes 2q + e).
  // Otherwise one 4-byte st.async per (peer, unit).
  const uint32_t hs_u = smem_u32(hs);
  const uint32_t bar_u = smem_u32(&bars[0]);
  constexpr int kMsgUnits = U == 2 ? 2 : 4;
  const bool vec = (Uc == U) && (((j0 + wu0) % kMsgUnits) == 0);
  const int vec_items = U == 8 ? 2 * C : C;
  uint32_t my_dst = 0, my_bar = 0;
  int my_src = 0;
  if (vec && lane < vec_items) {
    const int q = U == 8 ? lane >> 1 : lane;
    const int e = U == 8 ? (lane & 1) : 0;
    my_src = 4 * e;
    my_dst = map_to_rank(hs_u + (uint32_t)(j0 + wu0 + 4 * e) * 4u, (uint32_t)q);
    my_bar = map_to_rank(bar_u, (uint32_t)q);
  }
  // v: the value of lane u's unit; which = 0: h buffers / bars[buf];
  // which = 1: r.h buffers / bars[2 + buf]
  auto push = [&](float v, int which, int buf) {
    const uint32_t dshift = (which ? (uint32_t)((rhs - hs) * 4) : 0u) + (uint32_t)(buf * KP * 4);
    const uint32_t bshift = (uint32_t)((2 * which + buf) * sizeof(uint64_t));
    if (vec) {
      if constexpr (U == 2) {
        const float a = __shfl_sync(0xffffffffu, v, 0);
        const float c = __shfl_sync(0xffffffffu, v, 1);
        if (lane < vec_items) st_async_v2(my_dst + dshift, a, c, my_bar + bshift);
      } else {
        float4 x;
        x.x = __shfl_sync(0xffffffffu, v, (my_src + 0) & 31);
        x.y = __shfl_sync(0xffffffffu, v, (my_src + 1) & 31);
        x.z = __shfl_sync(0xffffffffu, v, (my_src + 2) & 31);
        x.w = __shfl_sync(0xffffffffu, v, (my_src + 3) & 31);
        if (lane < vec_items) st_async_v4(my_dst + dshift, x, my_bar + bshift);
      }
    } else {
      const int total = C * Uc;
      for (int i0 = 0; i0 < total; i0 += 32) {
        const int i = i0 + lane;
        const int q = Uc ? i / Uc : 0, u = Uc ? i % Uc : 0;
        const float x = __shfl_sync(0xffffffffu, v, u & 31);
        if (i < total)
          st_async_b32(map_to_rank(hs_u + (uint32_t)(j0 + wu0 + u) * 4u, (uint32_t)q) + dshift, x,
                       map_to_rank(bar_u, (uint32_t)q) + bshift);
      }
    }
  };

  // Bounded wait; false when this CTA gave up (then the warp leaves the loop).
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    if (abort_flag) return false;
    if (!mbar_wait_bounded(a, parity, p.timeout_ns)) {
      abort_flag = 1;
      atomicOr(p.status, 1);
      return false;
    }
    return true;
  };

  // xw of this lane's unit for step s (loaded one step ahead):
  // element (t, g) = xw_base + t * xw_tstride + g * H
  const size_t xw_tstride = p.layout == 0 ? (size_t)p.N * GH : GH;
  const float* xw_base = p.xw + xw_index(p, d, 0, b, 0, uj);
  auto load_xw = [&](int s, float (&x)[G]) {
    const bool on = gl && s < len && s < Tn;
    const float* q = xw_base + (size_t)(reverse ? len - 1 - s : s) * xw_tstride;
#pragma unroll
    // a coherent load: the projection may still have been running when this
    // kernel started, and a read-only-path load could be moved ahead of the
    // dependency wait
    for (int g = 0; g < G; ++g) x[g] = on ? __ldcg(q + (size_t)g * H) : 0.0f;
  };

  const uint32_t h_bytes = (uint32_t)H * 4u;
  if (tid == 0) {
    if (Tn > 1) mbar_arrive_expect_tx(smem_u32(&bars[1]), h_bytes);
    if (lbr0 && Tn > 0) mbar_arrive_expect_tx(smem_u32(&bars[2]), h_bytes);
  }
  // The launch may overlap the projection that writes Xw (programmatic
  // dependent launch): everything above only reads operands the projection
  // does not touch; wait for it before the first Xw read.
  grid_dependency_wait();
  // xw of the next two steps in flight: the load issued at the end of step s
  // is used at step s + 2.  One step ahead was too little for the direction
  // whose Xw rows sit in the other die's L2 (its row sums waited on the load:
  // about 1,450 against 1,190 cycles per step on the bidirectional 80 x 1 x
  // 256 layer), and a copy between two register sets would wait on it too,
  // so even and odd steps each keep their own set.  The variants with the
  // longest rows of R (KV = 4) keep one step ahead: two sets and the
  // unrolled loop would spill there.
  constexpr bool XW2 = KV <= 2;
  constexpr int kAhead = XW2 ? 2 : 1;
  float xa[G], xb[G];
  load_xw(0, xa);
  if constexpr (XW2) load_xw(1, xb);

  // ---------------- the steps
  // one step; xv holds step s's xw and is refilled with step s + kAhead's;
  // false when a wait gave up (the warp leaves the loop)
  auto step = [&](int s, float (&xv)[G]) -> bool {
    const int cur = s & 1, nxt = cur ^ 1;
    if (s >= 1 && !wait(&bars[cur], (uint32_t)(((s - 1) >> 1) & 1))) return false;
    // h_s has arrived, so every warp of every CTA is past step s-1: the fills
    // h_{s-1} of bars[nxt] and r.h_{s-1} of bars[2 + nxt] are complete and
    // the next ones can be announced
    if (tid == 0 && s + 1 < Tn) {
      if (s >= 1) mbar_arrive_expect_tx(smem_u32(&bars[nxt]), h_bytes);
      if (lbr0) mbar_arrive_expect_tx(smem_u32(&bars[2 + nxt]), h_bytes);
    }
    const bool active = s < len;
    const int t = active ? (reverse ? len - 1 - s : s) : s;
    const int ul = lane & (U - 1);  // the unit whose gates this lane gathers
    float hn = hreg;
    if constexpr (CELL == 1) {
      if (lbr0) {
        // z and r rows against h_prev; exchange r (.) h_prev; h rows against it
        const float v1 = rowsums<0, 2 * U, T, KV>(Rr, hs + (size_t)cur * KP, lane);
        const float sz = __shfl_sync(0xffffffffu, v1, row_lane<2 * U>(0 * U + ul));
        const float sr = __shfl_sync(0xffffffffu, v1, row_lane<2 * U>(1 * U + ul));
        const float z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, ((xv[0] + sz) + wbv[0]) + rbv[0]));
        const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, ((xv[1] + sr) + wbv[1]) + rbv[1]));
        push(r * hreg, 1, cur);
        if (!wait(&bars[2 + cur], (uint32_t)((s >> 1) & 1))) return false;
        const float v2 = rowsums<2 * U, U, T, KV>(Rr, rhs + (size_t)cur * KP, lane);
        const float sh = __shfl_sync(0xffffffffu, v2, row_lane<U>(ul));
        const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ((xv[2] + sh) + wbv[2]) + rbv[2]));
        if (active) hn = (1.0f - z) * hc + z * hreg;
      } else {
        const float v = rowsums<0, RW, T, KV>(Rr, hs + (size_t)cur * KP, lane);
        float sum[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sum[g] = __shfl_sync(0xffffffffu, v, row_lane<RW>(g * U + ul));
        const float z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, ((xv[0] + sum[0]) + wbv[0]) + rbv[0]));
        const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, ((xv[1] + sum[1]) + wbv[1]) + rbv[1]));
        const float ph = (xv[2] + r * (sum[2] + rbv[2])) + wbv[2];
        const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ph));
        if (active) hn = (1.0f - z) * hc + z * hreg;
      }
    } else {
      float v;
      if constexpr (GROUPED) v = rowsums_grouped<NRG, T, NCH>(Rg, hs + (size_t)cur * KP, lane);
      else v = rowsums<0, RW, T, KV>(Rr, hs + (size_t)cur * KP, lane);
      float pre[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float sum = __shfl_sync(0xffffffffu, v, GROUPED ? group_row_lane<NRG>(g * U + ul) : row_lane<RW>(g * U + ul));
        pre[g] = ((xv[g] + sum) + wbv[g]) + rbv[g];
      }
      if constexpr (CELL == 0) {
        float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
        if (has_p) {
          pi = pi + ppv[0] * creg;
          pf = pf + ppv[2] * creg;
        }
        const float ig = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pi));
        const float fg = input_forget ? 1.0f - ig : act<GEN, 0>(p, d * A + 0, clip_pre(clip, pf));
        const float cg = act<GEN, 1>(p, d * A + 1, clip_pre(clip, pc));
        const float cn = fg * creg + ig * cg;
        if (has_p) po = po + ppv[1] * cn;
        const float og = act<GEN, 0>(p, d * A + 0, clip_pre(clip, po));
        if (active) {
          hn = og * act<GEN, 1>(p, d * A + 2, cn);
          creg = cn;
        }
      } else {
        if (active) hn = act<GEN, 1>(p, d * A + 0, clip_pre(clip, pre[0]));
      }
    }
    hreg = hn;
    if (s + 1 < Tn) push(hn, 0, nxt);
    if (ybase != nullptr) store_elem<T>(ybase + (size_t)t * ystride, active ? hn : 0.0f);
    load_xw(s + kAhead, xv);
    return true;
  };
  if constexpr (XW2) {
    for (int s = 0; s < Tn; s += 2) {
      if (!step(s, xa)) break;
      if (s + 1 < Tn && !step(s + 1, xb)) break;
    }
  } else {
    for (int s = 0; s < Tn; ++s)
      if (!step(s, xa)) break;
  }

  // ---------------- outputs: zero Y past the loop, final states
  if (gl && !abort_flag) {
    if (ybase != nullptr)
      for (int t = Tn; t < S; ++t) store_elem<T>(ybase + (size_t)t * ystride, 0.0f);
    const bool zero = S > 0 && len == 0;
    const size_t si = state_index(p, d, b, uj);
    if (p.Yh != nullptr) store_elem<T>(static_cast<T*>(p.Yh) + si, zero ? 0.0f : hreg);
    if (CELL == 0 && p.Yc != nullptr) store_elem<T>(static_cast<T*>(p.Yc) + si, zero ? 0.0f : creg);
  }
  __syncthreads();
  cluster_sync_all();
}

// ------------------------------------------------------------------ launch
template <int CELL, typename T, bool GEN, int KV, int U, bool PLAIN>
cudaError_t step_fast_launch_one(const StepParams& p, const StepPlan& plan, cudaStream_t stream, int* resident) {
  auto kern = step_fast_kernel<CELL, T, GEN, KV, U, PLAIN>;
  if (plan.threads > (U == 2 ? 512 : 256) || plan.threads % 32 != 0) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.team_ctas > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)plan.team_ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the projection (the previous kernel on the stream) runs;
  // the kernel waits for it before reading Xw
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = resident != nullptr ? 1 : 2;
  if (resident != nullptr) {
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    *resident = (e == cudaSuccess) ? n : 0;
    return e;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Units per warp: RNN 8; LSTM and GRU 4 when a warp's 16 rows of R fit its
// registers (KV <= 2), else 2.
template <int CELL, int KV>
struct FastU {
  static constexpr int value = CELL == 2 ? 8 : (KV <= 2 ? 4 : 2);
};

template <int CELL, typename T, bool GEN, bool PLAIN>
cudaError_t step_fast_kv(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  switch (plan.kv) {
    case 1: return step_fast_launch_one<CELL, T, GEN, 1, FastU<CELL, 1>::value, PLAIN>(p, plan, s, q);
    case 2: return step_fast_launch_one<CELL, T, GEN, 2, FastU<CELL, 2>::value, PLAIN>(p, plan, s, q);
    case 4:
      if constexpr (sizeof(T) == 2) return step_fast_launch_one<CELL, T, GEN, 4, FastU<CELL, 4>::value, PLAIN>(p, plan, s, q);
      break;
    default: break;
  }
  return cudaErrorInvalidConfiguration;
}

// Units per warp the kernel of a plan uses (for the planner's thread count).
inline int fast_units_per_warp(int cell, int kv) { return cell == 2 ? 8 : (kv <= 2 ? 4 : 2); }

template <int CELL, typename T>
cudaError_t step_fast_dtype(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  const bool plain = !(p.clip > 0.0f) && p.P == nullptr && !p.input_forget;
  if (p.generic_acts) return plain ? step_fast_kv<CELL, T, true, true>(p, plan, s, q) : step_fast_kv<CELL, T, true, false>(p, plan, s, q);
  return plain ? step_fast_kv<CELL, T, false, true>(p, plan, s, q) : step_fast_kv<CELL, T, false, false>(p, plan, s, q);
}

template <int CELL>
cudaError_t step_fast_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  if (p.dtype == 0) return step_fast_dtype<CELL, float>(p, plan, s, q);
  if (p.dtype == 2) return step_fast_dtype<CELL, __nv_bfloat16>(p, plan, s, q);
  return step_fast_dtype<CELL, __half>(p, plan, s, q);
}

}  // namespace rk
