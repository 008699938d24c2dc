// rk_step_tcs.cu -- tensor-core recurrent step for small batches (at most 16
// rows per direction) of Half layers whose hidden units fit one cluster.
//
// Same arithmetic as rk_step.cuh and rk_step_tc.cuh (web page "Recurrent
// layers", sections "How a layer runs" and "Arithmetic and determinism"):
// per step and gate row pre = ((xw + rec) + Wb) + Rb with rec = R_row .
// h_prev (h rounded to Half for the product, state float32), then
// peepholes, clip, activation and state update (LSTM, RNN, GRU with
// linear_before_reset = 1).
//
// With a small batch the product is turned around: the MMA's M = 128 rows
// are this CTA's gate rows (row g * 32 + u for gate g, unit u of its 32
// units; rows past G * 32 are zero) held in shared memory for the whole
// layer, and its N = 16 columns are the direction's batch rows, so the
// exchanged operand is only 16 rows of h (2 KB per 64 k).  A team is one
// direction, one cluster of ceil(H / 32) CTAs.  Per step:
//   1. the producer warp waits until every CTA of the cluster has published
//      h_s (remote mbarrier arrivals, cluster-scope release / acquire) and
//      copies the direction's whole Half h_s (H / 64 blocks of 16 rows x 64
//      k, 128-byte swizzled, double-buffered in global memory) with one
//      bulk copy;
//   2. one lane issues the H / 16 MMAs (kind::f16, M = 128, N = 16, K = 16)
//      into one fp32 TMEM accumulator (lane = gate row, column = batch row);
//   3. warp g < G reads gate g's lanes (unit = lane) and stages them in
//      shared memory; every gate thread then takes one (unit, batch row)
//      pair (two when the batch exceeds 8), does the gate arithmetic, writes
//      its Half h into the next global buffer and Y, and the CTA publishes.
// The summation order is fixed (k in increasing 16-wide steps), so runs are
// bit-identical.  Every wait is bounded; on expiry the kernel sets the
// status word, drains its copy and MMAs, frees its TMEM and returns.
#include "rk_step_tc.cuh"

namespace rk {

namespace {

constexpr int XN = 16;         // MMA N: a direction's batch rows, padded
constexpr int XJ = 32;         // hidden units per CTA
constexpr int XPAIRS = 2;      // (unit, batch row) pairs per gate thread at most
constexpr int XBLK_A = 128 * 128;  // bytes of one 64-k block of the gate rows
constexpr int XBLK_B = XN * 128;   // bytes of one 64-k block of h

// Shared memory: [gate rows: KB x 16 KB][h: KB x 2 KB][staged products
// [4][32][16] floats][barriers][biases]
struct XsSmem {
  size_t r, h, acc, bar, bias, total;
};
__host__ __device__ inline XsSmem xs_layout(int G, int H) {
  XsSmem L{};
  const int KB = (H + SK - 1) / SK;
  size_t o = 1024;  // room to align the dynamic base up to 1024 bytes
  L.r = o;    o += (size_t)KB * XBLK_A;
  L.h = o;    o += (size_t)KB * XBLK_B;
  L.acc = o;  o += (size_t)4 * XJ * XN * 4;
  L.bar = o;  o += 256;
  L.bias = o; o += (size_t)2 * 4 * XJ * 4 + 3 * XJ * 4;
  L.total = o;
  (void)G;
  return L;
}

// Element offset of (buffer, direction, batch row b, unit j) in the Half h
// copy: [2][D][KB blocks][16 rows x 64 k, swizzled].
__device__ __forceinline__ size_t xs_h_block(const StepParams& p, int buf, int d, int kb, int KB) {
  return (((size_t)buf * p.D + d) * KB + kb) * (size_t)(XBLK_B / 2);
}

template <int CELL, bool GEN, bool PLAIN>
__global__ void __launch_bounds__(STHREADS, 1) step_tcs_kernel(const StepParams p, __half* __restrict__ h16) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  constexpr uint32_t kTmemCols = 32;  // accumulator: 128 lanes x 16 columns
  extern __shared__ unsigned char tsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  const XsSmem L = xs_layout(G, p.H);
  unsigned char* sR = base + (L.r - 1024);
  unsigned char* sH = base + (L.h - 1024);
  float* sAcc = reinterpret_cast<float*>(base + (L.acc - 1024));  // [g][u][b]
  // full, done, free, staged, pub (gather), drain, cluster publication[2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (L.bar - 1024));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  float* wb_s = reinterpret_cast<float*>(base + (L.bias - 1024));  // [g * XJ + u]
  float* rb_s = wb_s + 4 * XJ;
  float* pp_s = rb_s + 4 * XJ;                                     // [u * 3 + g]
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, N = p.N, S = p.S, Tn = p.T;
  const int C = p.team_ctas;
  const int d = blockIdx.x / C;  // one team (cluster) per direction
  int rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int j0 = rank * XJ;
  const int KB = (H + SK - 1) / SK;
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const size_t GH = (size_t)G * H;
  const __half* R = static_cast<const __half*>(p.R);
  const __half* Bias = static_cast<const __half*>(p.Bias);
  const __half* P = static_cast<const __half*>(p.P);
  const __half* h0 = static_cast<const __half*>(p.h0);
  const __half* c0 = static_cast<const __half*>(p.c0);
  __half* Y = static_cast<__half*>(p.Y);

  // ---------------- prologue: gate rows (row g * 32 + u), 16 bytes at a time
  const bool r_vec = (reinterpret_cast<uintptr_t>(R) & 15) == 0;
  for (int e = tid; e < KB * 128 * (SK / 8); e += blockDim.x) {
    const int kb = e / (128 * (SK / 8));
    const int rem = e % (128 * (SK / 8));
    const int r = rem / (SK / 8), kk = (rem % (SK / 8)) * 8;
    const int g = r / XJ, u = r % XJ, k = kb * SK + kk;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (g < G && j0 + u < H && k < H) {
      const __half* src = R + ((size_t)d * GH + (size_t)g * H + j0 + u) * H + k;
      if (r_vec) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        __align__(16) __half t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = src[i];
        v = *reinterpret_cast<const uint4*>(t8);
      }
    }
    *reinterpret_cast<uint4*>(sR + (size_t)kb * XBLK_A + sw128_offset(r, kk)) = v;
  }
  for (int e = tid; e < G * XJ; e += blockDim.x) {
    const int g = e / XJ, u = e % XJ;
    const bool ok = j0 + u < H && Bias != nullptr;
    wb_s[e] = ok ? __half2float(Bias[(size_t)d * 2 * GH + (size_t)g * H + j0 + u]) : 0.0f;
    rb_s[e] = ok ? __half2float(Bias[(size_t)d * 2 * GH + GH + (size_t)g * H + j0 + u]) : 0.0f;
  }
  for (int e = tid; e < 3 * XJ; e += blockDim.x) {
    const int u = e / 3, g = e % 3;
    pp_s[e] = (CELL == 0 && !PLAIN && P != nullptr && j0 + u < H) ? __half2float(P[(size_t)d * 3 * H + (size_t)g * H + j0 + u]) : 0.0f;
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);               // h copy landed
    mbar_init(smem_u32(&bars[1]), 1);               // accumulator complete (MMA commit)
    mbar_init(smem_u32(&bars[2]), 8);               // accumulator read (8 gate warps)
    mbar_init(smem_u32(&bars[3]), 8);               // products staged (8 gate warps)
    mbar_init(smem_u32(&bars[4]), 8);               // h copies written (8 gate warps)
    mbar_init(smem_u32(&bars[5]), 1);               // final MMA drain
    mbar_init(smem_u32(&bars[6]), (unsigned)C);     // every CTA published h_s, s even
    mbar_init(smem_u32(&bars[7]), (unsigned)C);     // ... s odd
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the gate rows were written by ordinary stores; the tensor cores read them
  // through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // gate threads: pair i = tid + 256 k is (unit i % 32, batch row i / 32)
  const bool gate_warp = warp < 8;
  float hreg[XPAIRS], creg[XPAIRS];
  int lenv[XPAIRS];
  bool pv[XPAIRS];
  const int pu = tid & 31;  // the unit is the same for both pairs
  const int pj = j0 + pu;
#pragma unroll
  for (int k = 0; k < XPAIRS; ++k) {
    const int b = (tid + 256 * k) >> 5;
    pv[k] = gate_warp && b < N;
    hreg[k] = creg[k] = 0.0f;
    lenv[k] = Tn;
  }
  // address of (buffer, batch row b, unit j) in the Half h copy
  auto h16_at = [&](int buf, int b, int j) {
    return reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(h16 + xs_h_block(p, buf, d, j / SK, KB)) +
                                     sw128_offset(b, j % SK));
  };
#pragma unroll
  for (int k = 0; k < XPAIRS; ++k) {
    if (!pv[k]) continue;
    const int b = (tid + 256 * k) >> 5;
    if (p.lens != nullptr) {
      int len = p.lens[b];
      len = len < 0 ? 0 : (len > S ? S : len);
      lenv[k] = len > Tn ? Tn : len;
    }
    if (pj < H) {
      const size_t si = state_index(p, d, b, pj);
      hreg[k] = h0 != nullptr ? __half2float(h0[si]) : 0.0f;
      creg[k] = (CELL == 0 && c0 != nullptr) ? __half2float(c0[si]) : 0.0f;
    }
    *h16_at(0, b, pj) = __float2half_rn(pj < H ? hreg[k] : 0.0f);  // h_0 into buffer 0
  }
  // k columns past the last CTA's units (up to the 64-wide block) belong to
  // no CTA: zero them once in both buffers for every row (R is zero there
  // too, but a stale Inf or NaN times zero would not be)
  if (rank == C - 1) {
    const int pad = KB * SK - C * XJ;
    for (int e = tid; e < pad * XN * 2; e += blockDim.x) {
      const int k = C * XJ + e % pad, b = (e / pad) % XN, buf = e / (pad * XN);
      *h16_at(buf, b, k) = __float2half_rn(0.0f);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA's barriers are initialised before any remote arrival (all CTAs
  // of a cluster run at once and reach this point)
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const uint32_t tmem_acc = *tmem_slot;

  const uint32_t bar_full = su32(&bars[0]), bar_done = su32(&bars[1]), bar_free = su32(&bars[2]);
  const uint32_t bar_staged = su32(&bars[3]), bar_pub = su32(&bars[4]), bar_drain = su32(&bars[5]);
  const uint32_t bar_pubc = su32(&bars[6]);
  // gate warps: make this CTA's new h copies visible to the async proxy,
  // gather the 8 warps, then lane q of warp 0 arrives on CTA q's
  // publication barrier for h_s (one barrier per step parity: a CTA's
  // arrivals for h_{s+2} come after it saw every arrival for h_{s+1}, each
  // made after its sender's arrivals for h_s)
  auto publish = [&](unsigned value, uint32_t pub_parity) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_pub) : "memory");
    if (warp == 0 && lane < C) {
      if (bar_wait(bar_pub, pub_parity, p.timeout_ns)) {
        const uint32_t local = bar_pubc + 8u * ((value - 1u) & 1u);  // h_s, s = value - 1
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(map_to_rank(local, (uint32_t)lane))
                     : "memory");
      } else {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
    }
  };
  uint32_t pub_parity = 0;
  if (gate_warp) publish(1u, pub_parity++ & 1u);

  const size_t xw_tstride = p.layout == 0 ? (size_t)N * GH : GH;
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;

  if (warp == 8) {
    // ---------------- producer lane: the whole h_s in one bulk copy
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)KB * XBLK_B;
      int armed = -1;
      bool ok = true;
      for (int s = 0; s < Tn && ok; ++s) {
        if (abort_flag || !bar_wait_cluster(bar_pubc + 8u * (uint32_t)(s & 1), (uint32_t)((s >> 1) & 1), p.timeout_ns)) {
          ok = false;
          break;
        }
        // the publishers' generic-proxy stores, acquired above, are read by the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        bar_expect(bar_full, bytes);
        bulk_load(su32(sH), h16 + xs_h_block(p, s & 1, d, 0, KB), bytes, bar_full);
        armed = s & 1;
      }
      if (!ok) {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
      // drain: the copy this CTA issued last must land before it exits
      if (armed >= 0) bar_wait(bar_full, (uint32_t)armed, p.timeout_ns);
    }
  } else if (warp == 9) {
    // ---------------- MMA lane: acc[128 gate rows x 16 batch] = R_rows . h^T
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(XN);
      const uint64_t adesc0 = desc_sw128(su32(sR));
      const uint64_t bdesc0 = desc_sw128(su32(sH));
      constexpr uint64_t kK16 = 32 >> 4;
      bool ok = true;
      for (int s = 0; s < Tn && ok; ++s) {
        if (abort_flag || !bar_wait(bar_full, (uint32_t)(s & 1), p.timeout_ns)) {
          ok = false;
          break;
        }
        // the gate warps must have read the previous step's accumulator
        if (s > 0 && !bar_wait(bar_free, (uint32_t)((s - 1) & 1), p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint64_t ad = adesc0, bd = bdesc0;
        for (int kb = 0; kb < KB; ++kb, ad += XBLK_A >> 4, bd += XBLK_B >> 4) {
          tc_mma(tmem_acc, ad, bd, idesc, kb != 0 ? 1u : 0u);
          tc_mma(tmem_acc, ad + kK16, bd + kK16, idesc, 1u);
          tc_mma(tmem_acc, ad + 2 * kK16, bd + 2 * kK16, idesc, 1u);
          tc_mma(tmem_acc, ad + 3 * kK16, bd + 3 * kK16, idesc, 1u);
        }
        tc_commit(bar_done);  // accumulator of step s complete
      }
      if (!ok) {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
      // drain: every MMA this CTA issued completes before TMEM is freed
      tc_commit(bar_drain);
      bar_wait(bar_drain, 0u, p.timeout_ns);
    }
  } else {
    // ---------------- gate warps
    float xv[XPAIRS][G];
    auto load_xw = [&](int s) {
#pragma unroll
      for (int k = 0; k < XPAIRS; ++k) {
        const int b = (tid + 256 * k) >> 5;
        const bool on = pv[k] && s < lenv[k] && s < Tn && pj < H;
        const float* qx = p.xw + xw_index(p, d, 0, on ? b : 0, 0, on ? pj : 0) +
                          (size_t)(on ? (reverse ? lenv[k] - 1 - s : s) : 0) * xw_tstride;
#pragma unroll
        for (int g = 0; g < G; ++g) xv[k][g] = on ? __ldg(qx + (size_t)g * H) : 0.0f;
      }
    };
    load_xw(0);
    bool ok = true;
    for (int s = 0; s < Tn; ++s) {
      if (abort_flag || !bar_wait(bar_done, (uint32_t)(s & 1), p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp < G) {
        // warp g holds gate g of the 32 units (lane = unit), 16 batch columns
        uint32_t v[XN];
        tmem_ld<XN>(tmem_acc + ((uint32_t)(warp * 32) << 16), v);
        float4* dst = reinterpret_cast<float4*>(sAcc + ((size_t)warp * XJ + lane) * XN);
#pragma unroll
        for (int i = 0; i < XN / 4; ++i)
          dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                               __uint_as_float(v[4 * i + 3]));
      }
      // the accumulator may be overwritten by the next step's product; the
      // staged products are read by every gate warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_free) : "memory");
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_staged) : "memory");
      }
      if (!bar_wait(bar_staged, (uint32_t)(s & 1), p.timeout_ns)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int k = 0; k < XPAIRS; ++k) {
        if (!pv[k]) continue;
        const int b = (tid + 256 * k) >> 5;
        const bool active = s < lenv[k];
        const int t = active ? (reverse ? lenv[k] - 1 - s : s) : s;
        float rec[G], pre[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          rec[g] = sAcc[((size_t)g * XJ + pu) * XN + b];
          pre[g] = ((xv[k][g] + rec[g]) + wb_s[g * XJ + pu]) + rb_s[g * XJ + pu];
        }
        float hn = hreg[k];
        if constexpr (CELL == 0) {
          // gates i, o, f, c
          float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
          if (has_p) {
            pi = pi + pp_s[pu * 3 + 0] * creg[k];
            pf = pf + pp_s[pu * 3 + 2] * creg[k];
          }
          const float ig = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pi));
          const float fg = input_forget ? 1.0f - ig : act<GEN, 0>(p, d * A + 0, clip_pre(clip, pf));
          const float cg = act<GEN, 1>(p, d * A + 1, clip_pre(clip, pc));
          const float cn = fg * creg[k] + ig * cg;
          if (has_p) po = po + pp_s[pu * 3 + 1] * cn;
          const float og = act<GEN, 0>(p, d * A + 0, clip_pre(clip, po));
          if (active) {
            hn = og * act<GEN, 1>(p, d * A + 2, cn);
            creg[k] = cn;
          }
        } else if constexpr (CELL == 1) {
          // linear_before_reset = 1: h~ = g((xw_h + r*(rec_h + Rb_h)) + Wb_h)
          const float z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[0]));
          const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[1]));
          const float ph = (xv[k][2] + r * (rec[2] + rb_s[2 * XJ + pu])) + wb_s[2 * XJ + pu];
          const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ph));
          if (active) hn = (1.0f - z) * hc + z * hreg[k];
        } else {
          if (active) hn = act<GEN, 1>(p, d * A + 0, clip_pre(clip, pre[0]));
        }
        if (pj < H) hreg[k] = hn;
        if (s + 1 < Tn) *h16_at((s + 1) & 1, b, pj) = __float2half_rn(pj < H ? hn : 0.0f);
        if (Y != nullptr && pj < H) Y[y_index(p, t, d, b, pj)] = __float2half_rn(active ? hn : 0.0f);
      }
      if (s + 1 < Tn) publish((unsigned)s + 2u, pub_parity++ & 1u);
      load_xw(s + 1);
    }
    if (!ok) {
      abort_flag = 1;
      atomicOr(p.status, 1);
    }
    // ---------------- outputs: zero Y past the loop, final states
    if (ok && !abort_flag && pj < H) {
#pragma unroll
      for (int k = 0; k < XPAIRS; ++k) {
        if (!pv[k]) continue;
        const int b = (tid + 256 * k) >> 5;
        if (Y != nullptr)
          for (int t = Tn; t < S; ++t) Y[y_index(p, t, d, b, pj)] = __float2half_rn(0.0f);
        const bool zero = S > 0 && lenv[k] == 0;
        const size_t si = state_index(p, d, b, pj);
        if (p.Yh != nullptr) static_cast<__half*>(p.Yh)[si] = __float2half_rn(zero ? 0.0f : hreg[k]);
        if (CELL == 0 && p.Yc != nullptr) static_cast<__half*>(p.Yc)[si] = __float2half_rn(zero ? 0.0f : creg[k]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_acc), "r"(kTmemCols) : "memory");
  }
  // no CTA leaves while a peer may still arrive on its barriers
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int CELL, bool GEN, bool PLAIN>
cudaError_t step_tcs_launch(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16) {
  auto kern = step_tcs_kernel<CELL, GEN, PLAIN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.team_ctas > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
  cfg.blockDim = dim3(STHREADS, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  // a team (direction) is one cluster; teams never wait on each other
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
  return cudaLaunchKernelEx(&cfg, kern, p, h16);
}

template <int CELL>
cudaError_t step_tcs_cell(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q, __half* h16) {
  const bool plain = !(p.clip > 0.0f) && p.P == nullptr && !p.input_forget;
  if (p.generic_acts)
    return plain ? step_tcs_launch<CELL, true, true>(p, plan, s, q, h16) : step_tcs_launch<CELL, true, false>(p, plan, s, q, h16);
  return plain ? step_tcs_launch<CELL, false, true>(p, plan, s, q, h16) : step_tcs_launch<CELL, false, false>(p, plan, s, q, h16);
}

}  // namespace

size_t step_tcs_smem(int G, int H) { return xs_layout(G, H).total; }

cudaError_t step_tcs_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16) {
  __half* hp = static_cast<__half*>(h16);
  switch (p.cell) {
    case 0: return step_tcs_cell<0>(p, plan, s, resident, hp);
    case 1: return step_tcs_cell<1>(p, plan, s, resident, hp);
    default: return step_tcs_cell<2>(p, plan, s, resident, hp);
  }
}

}  // namespace rk
