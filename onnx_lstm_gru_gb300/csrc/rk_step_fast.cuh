// rk_step_fast.cuh -- latency-first persistent step kernel for layers whose
// team holds one batch row: the projection is fused into the step kernel and
// R lives in registers.
//
// What it computes is the same as rk_step.cuh (web page "Recurrent layers",
// sections "How a layer runs" and "Arithmetic and determinism"): per step and
// gate row pre = ((xw + rec) + Wb) + Rb with xw = x_t . W_row and
// rec = R_row . h_prev, then peepholes, clip, activation and state update;
// GRU with linear_before_reset = 0 exchanges r (.) h_prev of every unit
// before the candidate's product.
//
// Layout of one CTA (one cluster of C CTAs per (direction, batch row)):
//   - J <= 32 hidden units per CTA, G*Jp rows (Jp = J rounded up to 8).
//   - "matvec" warps 0 .. MW-1: warp w keeps rows 8w .. 8w+7 of R for the
//     whole layer in registers (lanes hold k = 4*(32*chunk + lane) + e).  Per
//     step it reads h_prev from shared memory, chains each lane's terms in
//     increasing k and folds the 32 lane sums with the fixed shuffle tree.
//   - warp 0 also does the gate arithmetic: lane j owns unit j0 + j and keeps
//     its h, c, biases and peepholes in registers, writes Y and pushes the new
//     h (float4 groups gathered by shuffles) into every CTA of the cluster
//     with st.async; each receiver's mbarrier counts the bytes.
//   - "producer" warps (fused projection): compute xw for upcoming steps from
//     x_t (read from X as stored) and the CTA's rows of W (held in shared
//     memory) into a 4-slot ring guarded by full / empty mbarriers, running
//     ahead of the recurrence.  The projection's sums are lane-strided chains
//     folded by the same shuffle tree, so runs are bit-identical.
//   - named barriers (not CTA-wide ones) hand the row sums to warp 0, so the
//     other warps go straight on to the next step's wait.
// Every mbarrier wait is bounded by a deadline on %globaltimer.  When one
// gives up the CTA sets the status word and enters an abort mode in which no
// wait or push happens but every named barrier is still passed, so no warp
// can be left waiting; the kernel then winds down.
#pragma once

#include "rk_step.cuh"

namespace rk {

constexpr int kFastRing = 4;      // xw ring slots
constexpr int kFastProducers = 4; // producer warps when the projection is fused;
                                  // producer warp w owns steps w, w + 4, ... and ring slot w

struct FastSmem {
  size_t hs, rhs, gs, Ws, xws, stage, bar, total;
};

// Shared memory of the fast kernel (offsets in bytes).
__host__ __device__ inline FastSmem fast_smem_layout(const StepParams& p, int rows_pad, bool fused, int elem_bytes) {
  FastSmem L{};
  size_t o = 0;
  const bool lbr0 = p.cell == 1 && !p.lbr;
  L.hs = o;  o = align16(o + 2 * (size_t)p.KP * 4);
  L.rhs = o; o = align16(o + (lbr0 ? 2 * (size_t)p.KP * 4 : 0));
  L.gs = o;  o = align16(o + (size_t)rows_pad * 4);
  L.Ws = o;  o = align16(o + (fused ? (size_t)rows_pad * p.IP * elem_bytes : 0));
  L.xws = o; o = align16(o + (fused ? (size_t)kFastRing * rows_pad * 4 : 0));
  L.stage = o; o = align16(o + 2 * 32 * 4);
  L.bar = o; o = align16(o + (4 + 2 * kFastRing) * 8);
  L.total = o;
  return L;
}

// R fragment kept in registers: 4 consecutive k of one row.
template <typename T>
struct RFrag;
template <>
struct RFrag<float> {
  float4 v;
  __device__ __forceinline__ float4 get() const { return v; }
  __device__ __forceinline__ void set(const float e[4]) { v = make_float4(e[0], e[1], e[2], e[3]); }
};
template <>
struct RFrag<__half> {
  uint2 v;
  __device__ __forceinline__ float4 get() const {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ __forceinline__ void set(const float e[4]) {
    __half2 a = __floats2half2_rn(e[0], e[1]);
    __half2 b = __floats2half2_rn(e[2], e[3]);
    v.x = *reinterpret_cast<uint32_t*>(&a);
    v.y = *reinterpret_cast<uint32_t*>(&b);
  }
};

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Rows r0..r0+7 of a register-resident R fragment times h (KV float4 slices
// per lane); returns the lane's partial sum slot after the shuffle tree
// (valid for lanes with (lane & 3) == 0, row index xreduce_index<8>(lane)).
template <typename T, int KV>
__device__ __forceinline__ float rowsums_regs(const RFrag<T> (&R)[8][KV], const float* __restrict__ h, int lane) {
  float4 hv[KV];
#pragma unroll
  for (int kc = 0; kc < KV; ++kc) hv[kc] = *reinterpret_cast<const float4*>(h + (kc * 32 + lane) * 4);
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float a = 0.0f;
#pragma unroll
    for (int kc = 0; kc < KV; ++kc) {
      const float4 rv = R[r][kc].get();
      a = fmaf(rv.x, hv[kc].x, a);
      a = fmaf(rv.y, hv[kc].y, a);
      a = fmaf(rv.z, hv[kc].z, a);
      a = fmaf(rv.w, hv[kc].w, a);
    }
    acc[r] = a;
  }
  xreduce<8, 16>(acc, lane);
  return acc[0];
}

template <int CELL, typename T, bool GEN, int KV, bool FUSED>
__global__ void __launch_bounds__(512, 1) step_fast_kernel(const StepParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  constexpr int RING = kFastRing;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = p.team_ctas;
  const int rank = (int)cluster_ctarank();
  const int team = blockIdx.x / C;
  const int d = team / p.N, b = team % p.N;  // one batch row per team
  const int J = p.J, H = p.H, KP = p.KP, I = p.I, IP = p.IP;
  const int Jp = p.rows_pad / G;
  const int MW = p.rows_pad / 8;  // matvec warps
  const int j0 = rank * J;
  const int Jc = max(0, min(J, H - j0));
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const bool lbr0 = (CELL == 1) && !p.lbr;
  // GRU lbr = 0: rows [0, 2Jp) (z, r) form phase 1, rows [2Jp, 3Jp) phase 2
  const int MW1 = lbr0 ? (2 * Jp) / 8 : MW;
  const int n_bar1 = MW1 * 32;
  const int n_bar2 = ((lbr0 ? Jp / 8 : 0) + 1) * 32;
  const int S = p.S, Tn = p.T;

  const FastSmem L = fast_smem_layout(p, p.rows_pad, FUSED, (int)sizeof(T));
  float* hs = reinterpret_cast<float*>(smem + L.hs);
  float* rhs = reinterpret_cast<float*>(smem + L.rhs);
  float* gs = reinterpret_cast<float*>(smem + L.gs);
  T* Ws = reinterpret_cast<T*>(smem + L.Ws);
  float* xws = reinterpret_cast<float*>(smem + L.xws);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);  // h[2], rh[2], full[RING], empty[RING]
  __shared__ volatile int abort_flag;

  const T* R = static_cast<const T*>(p.R);
  const T* W = static_cast<const T*>(p.W);
  const T* X = static_cast<const T*>(p.X);
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

  // ---------------- prologue
  RFrag<T> Rr[8][KV];
  if (warp < MW) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int lr = warp * 8 + r, g = lr / Jp, jl = lr % Jp;
      const bool ok = g < G && jl < Jc;
      const T* row = R + ((size_t)d * GH + (size_t)g * H + j0 + jl) * H;
#pragma unroll
      for (int kc = 0; kc < KV; ++kc) {
        const int k = (kc * 32 + lane) * 4;
        float e[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) e[q] = (ok && k + q < H) ? load_elem<T>(row + k + q) : 0.0f;
        Rr[r][kc].set(e);
      }
    }
  }
  if constexpr (FUSED) {
    for (size_t e = tid; e < (size_t)p.rows_pad * IP; e += blockDim.x) {
      const int lr = (int)(e / IP), i = (int)(e % IP), g = lr / Jp, jl = lr % Jp;
      Ws[e] = (g < G && jl < Jc && i < I) ? W[((size_t)d * GH + (size_t)g * H + j0 + jl) * I + i]
                                          : static_cast<T>(0.0f);
    }
  }
  for (int e = tid; e < 2 * KP; e += blockDim.x) {
    const int k = e % KP;
    hs[e] = (e < KP && k < H && h0 != nullptr) ? load_elem<T>(h0 + state_index(p, d, b, k)) : 0.0f;
    if (lbr0) rhs[e] = 0.0f;
  }
  // gate-lane state (warp 0, lane j < Jc owns unit j0 + j)
  const bool gl = warp == 0 && lane < Jc;
  const int uj = j0 + lane;
  float hreg = 0.0f, creg = 0.0f, wbv[G], rbv[G], ppv[3];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    wbv[g] = (gl && Bias != nullptr) ? load_elem<T>(Bias + (size_t)d * 2 * GH + (size_t)g * H + uj) : 0.0f;
    rbv[g] = (gl && Bias != nullptr) ? load_elem<T>(Bias + (size_t)d * 2 * GH + GH + (size_t)g * H + uj) : 0.0f;
  }
#pragma unroll
  for (int g = 0; g < 3; ++g) ppv[g] = (CELL == 0 && gl && P != nullptr) ? load_elem<T>(P + (size_t)d * 3 * H + (size_t)g * H + uj) : 0.0f;
  const bool has_p = CELL == 0 && P != nullptr;
  if (gl) {
    const size_t si = state_index(p, d, b, uj);
    hreg = h0 != nullptr ? load_elem<T>(h0 + si) : 0.0f;
    creg = (CELL == 0 && c0 != nullptr) ? load_elem<T>(c0 + si) : 0.0f;
  }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(smem_u32(&bars[4 + i]), 1);
      mbar_init(smem_u32(&bars[4 + RING + i]), 1);
    }
    abort_flag = 0;
    fence_mbar_init_cluster();
  }
  cluster_sync_all();

  // Bounded wait; once any wait of this CTA gave up, waits return at once.
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return;
    if (abort_flag) return;
    if (!mbar_wait_bounded(a, parity, p.timeout_ns)) {
      abort_flag = 1;
      atomicOr(p.status, 1);
    }
  };

  // Warp 0 pushes the lane-held values of its units (lane j = unit j0 + j)
  // into every CTA of the cluster.  Item i = 32 m + lane is chunk c of peer q
  // (float4 chunks when J and H are multiples of 4, else single floats).  The
  // remote addresses of the first kPre items per lane are computed once here
  // (buffer 1 lies KP floats after buffer 0, bars[1] 8 bytes after bars[0]).
  const bool vec = ((J & 3) == 0) && ((H & 3) == 0);
  const int per_peer = vec ? (Jc >> 2) : Jc;
  const int n_items = C * per_peer;
  constexpr int kPre = 4;
  uint32_t it_dst[kPre], it_bar[kPre];
  int it_chunk[kPre];
  float* stage = reinterpret_cast<float*>(smem + L.stage);
#pragma unroll
  for (int m = 0; m < kPre; ++m) {
    const int i = m * 32 + lane;
    it_chunk[m] = -1;
    it_dst[m] = 0;
    it_bar[m] = 0;
    if (warp == 0 && i < n_items) {
      const int q = i / per_peer, c = i % per_peer;
      it_chunk[m] = c;
      it_dst[m] = map_to_rank(smem_u32(hs) + (uint32_t)(j0 + (vec ? 4 * c : c)) * 4u, (uint32_t)q);
      it_bar[m] = map_to_rank(smem_u32(&bars[0]), (uint32_t)q);
    }
  }
  // values v of lanes 0..Jc-1 into buffer `buf` of the h exchange (which = 0)
  // or of the r.h exchange (which = 1: rhs and bars[2 + buf])
  auto push = [&](float v, int which, int buf) {
    float* st = stage + which * 32;
    st[lane] = v;
    __syncwarp();
    if (abort_flag) return;
    const uint32_t dshift = (which ? (uint32_t)((rhs - hs) * 4) : 0u) + (uint32_t)(buf * KP * 4);
    const uint32_t bshift = (uint32_t)((2 * which + buf) * sizeof(uint64_t));
#pragma unroll
    for (int m = 0; m < kPre; ++m) {
      const int c = it_chunk[m];
      if (c >= 0) {
        if (vec) {
          st_async_v4(it_dst[m] + dshift, *reinterpret_cast<const float4*>(st + 4 * c), it_bar[m] + bshift);
        } else {
          st_async_b32(it_dst[m] + dshift, st[c], it_bar[m] + bshift);
        }
      }
    }
    for (int i = kPre * 32 + lane; i < n_items; i += 32) {  // more than kPre items per lane
      const int q = i / per_peer, c = i % per_peer;
      const uint32_t dst = map_to_rank(smem_u32(hs) + (uint32_t)(j0 + (vec ? 4 * c : c)) * 4u, (uint32_t)q) + dshift;
      const uint32_t bar = map_to_rank(smem_u32(&bars[0]), (uint32_t)q) + bshift;
      if (vec) {
        st_async_v4(dst, *reinterpret_cast<const float4*>(st + 4 * c), bar);
      } else {
        st_async_b32(dst, st[c], bar);
      }
    }
  };
  const uint32_t h_bytes = (uint32_t)H * 4u;

  if (warp < MW) {
    // ================= recurrence (matvec warps; warp 0 also gates and pushes)
    const bool phase1 = warp < MW1;
    // the thread that announces the bytes each exchange expects: off warp 0's
    // critical path when there is another phase-1 warp
    const int expect_tid = MW1 > 1 ? 32 : 0;
    // Y of this lane's unit: element (t, d, b, uj) = ybase + t * ystride
    const size_t ystride = p.layout == 0 ? (size_t)p.D * p.N * H : (size_t)p.D * H;
    T* ybase = (Y != nullptr && gl) ? Y + y_index(p, 0, d, b, uj) : nullptr;
    if (tid == expect_tid) {
      if (Tn > 1) mbar_arrive_expect_tx(smem_u32(&bars[1]), h_bytes);
      if (lbr0 && Tn > 0) mbar_arrive_expect_tx(smem_u32(&bars[2]), h_bytes);
    }
    for (int s = 0; s < Tn; ++s) {
      const int cur = s & 1, nxt = cur ^ 1;
      if (phase1) {
        if (s >= 1) wait(&bars[cur], (uint32_t)(((s - 1) >> 1) & 1));
        // h_s has arrived, so every CTA is past step s-1: the previous fills of
        // bars[nxt] (h_{s-1}) and of bars[2 + nxt] (r.h of step s-1) are
        // complete and the next ones can be announced: h_{s+1} (h_1 was
        // announced before the loop) and, for GRU lbr = 0, r.h of step s+1
        if (tid == expect_tid && s + 1 < Tn) {
          if (s >= 1) mbar_arrive_expect_tx(smem_u32(&bars[nxt]), h_bytes);
          if (lbr0) mbar_arrive_expect_tx(smem_u32(&bars[2 + nxt]), h_bytes);
        }
        const float v = rowsums_regs<T, KV>(Rr, hs + (size_t)cur * KP, lane);
        if ((lane & 3) == 0) gs[warp * 8 + xreduce_index<8>(lane)] = v;
        if (warp == 0) named_bar_sync(1, n_bar1); else named_bar_arrive(1, n_bar1);
      } else {
        // GRU lbr = 0, phase 2 rows: wait for r (.) h_prev of every unit
        wait(&bars[2 + cur], (uint32_t)((s >> 1) & 1));
        const float v = rowsums_regs<T, KV>(Rr, rhs + (size_t)cur * KP, lane);
        if ((lane & 3) == 0) gs[warp * 8 + xreduce_index<8>(lane)] = v;
        named_bar_arrive(2, n_bar2);
      }
      if (warp != 0) continue;

      // ---- warp 0: gate arithmetic of this step
      const int slot = s % RING;
      const bool active = s < len;
      const int t = active ? (reverse ? len - 1 - s : s) : s;
      float xv[G];
      if constexpr (FUSED) {
        wait(&bars[4 + slot], (uint32_t)((s / RING) & 1));
#pragma unroll
        for (int g = 0; g < G; ++g) xv[g] = gl ? xws[slot * p.rows_pad + g * Jp + lane] : 0.0f;
        __syncwarp();
        if (lane == 0) mbar_arrive_local(smem_u32(&bars[4 + RING + slot]));
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) xv[g] = (gl && active) ? __ldg(p.xw + xw_index(p, d, t, b, g, uj)) : 0.0f;
      }
      float pre[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pre[g] = gl ? ((xv[g] + gs[g * Jp + lane]) + wbv[g]) + rbv[g] : 0.0f;
      float hn = hreg;
      if constexpr (CELL == 0) {
        float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
        if (has_p) {
          pi = pi + ppv[0] * creg;
          pf = pf + ppv[2] * creg;
        }
        const float ig = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pi));
        const float fg = p.input_forget ? 1.0f - ig : act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pf));
        const float cg = act<GEN, 1>(p, d * A + 1, clip_pre(p.clip, pc));
        const float cn = fg * creg + ig * cg;
        if (has_p) po = po + ppv[1] * cn;
        const float og = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, po));
        if (active) {
          hn = og * act<GEN, 1>(p, d * A + 2, cn);
          creg = cn;
        }
      } else if constexpr (CELL == 1) {
        const float z = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pre[0]));
        const float r = act<GEN, 0>(p, d * A + 0, clip_pre(p.clip, pre[1]));
        float ph;
        if (lbr0) {
          // exchange r (.) h_prev, then the phase-2 warps form R_h . (r (.) h_prev)
          push(r * hreg, 1, cur);
          named_bar_sync(2, n_bar2);
          ph = gl ? ((xv[2] + gs[2 * Jp + lane]) + wbv[2]) + rbv[2] : 0.0f;
        } else {
          ph = gl ? (xv[2] + r * (gs[2 * Jp + lane] + rbv[2])) + wbv[2] : 0.0f;
        }
        const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(p.clip, ph));
        if (active) hn = (1.0f - z) * hc + z * hreg;
      } else {
        if (active) hn = act<GEN, 1>(p, d * A + 0, clip_pre(p.clip, pre[0]));
      }
      hreg = hn;
      if (ybase != nullptr) store_elem<T>(ybase + (size_t)t * ystride, active ? hn : 0.0f);
      if (s + 1 < Tn) push(hn, 0, nxt);
    }
  } else if (FUSED && warp < MW + kFastProducers) {
    // ================= producers: xw for upcoming steps into the ring
    static_assert(kFastRing == kFastProducers, "one ring slot per producer warp");
    const int pw = warp - MW;
    const int nrg = p.rows_pad / 8;
    const int nic = IP / kKChunk;
    for (int s = pw; s < Tn; s += kFastProducers) {
      const int slot = s % RING, n = s / RING;
      if (n >= 1) wait(&bars[4 + RING + slot], (uint32_t)((n - 1) & 1));
      const int t = s < len ? (reverse ? len - 1 - s : s) : s;
      const T* xrow = X + (p.layout == 0 ? ((size_t)t * p.N + b) : ((size_t)b * S + t)) * I;
      for (int rg = 0; rg < nrg; ++rg) {
        float acc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
        for (int ic = 0; ic < nic; ++ic) {
          const int i = (ic * 32 + lane) * 4;
          float xe[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) xe[q] = i + q < I ? load_elem<T>(xrow + i + q) : 0.0f;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float4 wv = load4_smem<T>(Ws + (size_t)(rg * 8 + r) * IP + i);
            float a = acc[r];
            a = fmaf(wv.x, xe[0], a);
            a = fmaf(wv.y, xe[1], a);
            a = fmaf(wv.z, xe[2], a);
            a = fmaf(wv.w, xe[3], a);
            acc[r] = a;
          }
        }
        xreduce<8, 16>(acc, lane);
        if ((lane & 3) == 0) xws[slot * p.rows_pad + rg * 8 + xreduce_index<8>(lane)] = acc[0];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(smem_u32(&bars[4 + slot]));
    }
  }

  // ---------------- outputs: zero Y past the loop, final states
  if (gl && !abort_flag) {
    if (Y != nullptr)
      for (int t = Tn; t < S; ++t) store_elem<T>(Y + y_index(p, t, d, b, uj), 0.0f);
    const bool zero = S > 0 && len == 0;
    const size_t si = state_index(p, d, b, uj);
    if (p.Yh != nullptr) store_elem<T>(static_cast<T*>(p.Yh) + si, zero ? 0.0f : hreg);
    if (CELL == 0 && p.Yc != nullptr) store_elem<T>(static_cast<T*>(p.Yc) + si, zero ? 0.0f : creg);
  }
  __syncthreads();
  cluster_sync_all();
}

// ------------------------------------------------------------------ launch
template <int CELL, typename T, bool GEN, int KV, bool FUSED>
cudaError_t step_fast_launch_one(const StepParams& p, const StepPlan& plan, cudaStream_t stream, int* resident) {
  auto kern = step_fast_kernel<CELL, T, GEN, KV, FUSED>;
  if (plan.threads > 512 || plan.threads % 32 != 0) return cudaErrorInvalidConfiguration;
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)plan.team_ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (resident != nullptr) {
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    *resident = (e == cudaSuccess) ? n : 0;
    return e;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CELL, typename T, bool GEN, bool FUSED>
cudaError_t step_fast_kv(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  switch (plan.kv) {
    case 1: return step_fast_launch_one<CELL, T, GEN, 1, FUSED>(p, plan, s, q);
    case 2: return step_fast_launch_one<CELL, T, GEN, 2, FUSED>(p, plan, s, q);
    case 4:
      if constexpr (sizeof(T) == 2) return step_fast_launch_one<CELL, T, GEN, 4, FUSED>(p, plan, s, q);
      break;
    default: break;
  }
  return cudaErrorInvalidConfiguration;
}

template <int CELL>
cudaError_t step_fast_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  const bool gen = p.generic_acts != 0;
  if (p.dtype == 0) {
    if (plan.fused) return gen ? step_fast_kv<CELL, float, true, true>(p, plan, s, q) : step_fast_kv<CELL, float, false, true>(p, plan, s, q);
    return gen ? step_fast_kv<CELL, float, true, false>(p, plan, s, q) : step_fast_kv<CELL, float, false, false>(p, plan, s, q);
  }
  if (plan.fused) return gen ? step_fast_kv<CELL, __half, true, true>(p, plan, s, q) : step_fast_kv<CELL, __half, false, true>(p, plan, s, q);
  return gen ? step_fast_kv<CELL, __half, true, false>(p, plan, s, q) : step_fast_kv<CELL, __half, false, false>(p, plan, s, q);
}

}  // namespace rk
