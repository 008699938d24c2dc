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
//     goes to a double-buffered global array (L2 resident) and each CTA
//     raises the team's counter with a release add.  A staging warp per CTA
//     polls the counter with acquire loads from the moment its CTA's products
//     are done (while the other warps do the gate arithmetic) and bulk-copies
//     the rows into shared memory as soon as every CTA has published; the
//     other warps wait only for the copies to land.  No CTA barrier spans the
//     team's exchange.
// Every wait is bounded by a deadline on %globaltimer; a wait that runs out
// sets bit 0 of the status word and the kernel winds down without hanging.
#pragma once

#include "rk_step_common.cuh"

namespace rk {

// Row sums gs[(row0 + r) * gs_ld + col0 + b] = sum_k Rs[row0 + r][k] * hsrc[b][k]
// for rows [row0, row0 + nrows) (nrows a multiple of RPW) and NBC batch rows.
template <int RPW, int NBC, typename T, int UNROLL = 1>
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
#pragma unroll UNROLL
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
// Shared-memory layout of one CTA (all offsets in bytes, 16-byte aligned).
struct SmemLayout {
  size_t Rs, hs, rhs, gs, hown, cs, zs, stage, rstage, wb, rb, pp, lens, xs, bar, total;
};


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
  L.xs = o;   o = align16(o + (size_t)nb * p.J * p.G * 4);  // each pair's Xw of the step (prefetched)
  L.bar = o;  o = align16(o + 4 * 8);
  L.total = o;
  return L;
}

// Threads per CTA the kernel is compiled for (registers are budgeted for it:
// the grid kernel's 32-value tiles get 96 registers a thread, room for the
// staging warp's state without spilling the tile).
template <int RPW, int NBC, bool GRID>
struct MaxThreads {
  static constexpr int value = (RPW * NBC >= 32) ? (GRID ? 640 : 768) : (GRID ? 320 : 512);
};

template <int CELL, typename T, bool GEN, int RPW, int NBC, bool GRID>
__global__ void __launch_bounds__(MaxThreads<RPW, NBC, GRID>::value, 1) step_kernel(const StepParams p) {
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
  // the direction's activation slots f, g, h (generic activations), read once
  ActSlot af{}, ag{}, ah{};
  if constexpr (GEN) {
    af = p.acts[d * A + 0];
    if constexpr (A > 1) ag = p.acts[d * A + 1];
    if constexpr (A > 2) ah = p.acts[d * A + 2];
  }
  // grid kernel: the last warp stages the exchanged rows, the others compute
  // (tid_c: the thread's index among the computing threads, past every pair
  // for the staging warp)
  const bool producer = GRID && warp == nwarps - 1;
  const int NTc = GRID ? NT - 32 : NT;
  const int tid_c = producer ? (1 << 30) : tid;
  // grid kernel: the team's release counters for h and for r.h, each on a
  // 128-byte line of its own
  unsigned* ctr_h = GRID ? p.team_ctrs + (size_t)team * kGridCounterWordsPerTeam : nullptr;
  unsigned* ctr_rh = GRID ? ctr_h + 32 : nullptr;

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
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  // cluster: [0,1] h buffers, [2,3] r.h buffers; grid: [0] staged rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);

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
      if (tid == 0) {
        mbar_init(smem_u32(&bars[0]), 1);  // staged rows landed
        fence_mbar_init_cluster();
      }
      // the exchange buffer is written by ordinary stores and read by bulk copies
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }

  uint32_t stage_no = 0;  // grid: stagings of exchanged rows so far (each completes mbarrier bars[0] once)
  bool alive = true;
  // grid: this CTA's new h (or r.h) is in the exchange buffer: one release add
  // on the team's counter (after a barrier that orders the writing threads'
  // stores and proxy fences before it)
  auto publish = [&](unsigned* ctr) { asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory"); };
  if constexpr (GRID) {
    __syncthreads();
    if (tid == 0) publish(ctr_h);
  }

  // Grid kernel, staging warp: copy batch rows [c0, c0 + NBC) of an exchange
  // buffer into hs, completing mbarrier bars[0].  With `ctr`, lane 0 first
  // waits until the team's counter shows every CTA's publication number
  // `want`.  Rows of a whole number of 16 bytes: one bulk copy per row.  Other
  // rows: element loads by the whole warp.  A wait that gives up still
  // completes the mbarrier (with a plain arrival) so that no reader waits on
  // it, and returns false.  Rows past the team's batch keep stale values whose
  // sums no gate reads; columns past H stay zero from the prologue.
  const bool bulk_rows = (H % 4) == 0;
  auto stage_rows = [&](const float* src, int c0, const unsigned* ctr, unsigned want) -> bool {
    const int nr = min(NBC, nbt - c0);
    const float* rows = src + ((size_t)d * p.N + b0 + c0) * KP;
    const uint32_t bar = smem_u32(&bars[0]);
    int rdy = 1;
    if (lane == 0 && ctr != nullptr) rdy = counter_wait_bounded(ctr, (unsigned)C * want, p.timeout_ns) ? 1 : 0;
    // also orders lane 0's acquire before the other lanes' loads
    const bool ok = __shfl_sync(0xffffffffu, rdy, 0) != 0;
    if (!ok) {
      if (lane == 0) mbar_arrive(bar);
      return false;
    }
    if (bulk_rows) {
      if (lane == 0) {
        // the writers' stores (made visible to the async proxy before their
        // release) are read by the async proxy; this CTA's earlier reads of
        // hs come before the async proxy rewrites it
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, (uint32_t)nr * (uint32_t)H * 4u);
        for (int bl = 0; bl < nr; ++bl)
          bulk_copy_g2s(smem_u32(hs + (size_t)bl * KP), rows + (size_t)bl * KP, (uint32_t)H * 4u, bar);
      }
      return true;
    }
    for (int e = lane; e < nr * H; e += 32) {
      const int bl = e / H, k = e % H;
      hs[(size_t)bl * KP + k] = __ldcg(rows + (size_t)bl * KP + k);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    return true;
  };

  // Row sums for rows [row0, row0 + nrows) against the current h (or r.h).
  // Cluster kernel: h is already in shared memory.  Grid kernel: per chunk of
  // NBC batch rows the staging warp copies the rows (waiting for the team's
  // counter on the first chunk; it starts while the other warps still do the
  // previous phase's gate arithmetic) and the other warps multiply them once
  // landed; a barrier of the whole CTA ends every chunk.  Returns false (grid
  // kernel, every thread alike) when a wait gave up.
  auto products = [&](int row0, int nrows, const float* cluster_src, const float* global_src, const unsigned* ctr,
                      unsigned want) -> bool {
    if constexpr (!GRID) {
      matvec<RPW, NBC, T>(Rs, KP, row0, nrows, cluster_src, gs, NBC, 0, warp, nwarps, lane);
      return true;
    } else {
      for (int c0 = 0; c0 < nbt; c0 += NBC) {
        bool ok;
        if (producer) {
          ok = stage_rows(global_src, c0, c0 == 0 ? ctr : nullptr, want);
        } else {
          ok = mbar_wait_bounded(smem_u32(&bars[0]), stage_no & 1u, p.timeout_ns);
          matvec<RPW, NBC, T, (RPW * NBC >= 32) ? 1 : 2>(Rs, KP, row0, nrows, hs, gs, nb_ld, c0, warp, nwarps - 1, lane);
        }
        ++stage_no;
        if (__syncthreads_or(!ok)) {
          if (tid == 0) atomicOr(p.status, 1);
          return false;
        }
      }
      return true;
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
  // The thread's first (unit, batch row) pair, whose indices every step
  // reuses: unit fj, row fb, its Y index at t = 0 (Y advances by y_tstride
  // per time step) and its index in an exchange buffer.
  const int fj = tid_c < npairs ? tid_c % Jc : 0, fb = tid_c < npairs ? tid_c / Jc : 0;
  const size_t fy0 = y_index(p, 0, d, b0 + fb, j0 + fj);
  const size_t y_tstride = p.layout == 0 ? (size_t)p.D * p.N * H : (size_t)p.D * H;
  const size_t fg0 = ((size_t)d * p.N + b0 + fb) * KP + j0 + fj;
  const size_t hbuf = (size_t)p.D * p.N * KP;  // floats per exchange buffer
  // the first pair's biases and peepholes, held in registers for the launch
  float fwb[G], frb[G], fpp[3];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    fwb[g] = wb_s[g * Jp + fj];
    frb[g] = rb_s[g * Jp + fj];
  }
#pragma unroll
  for (int q = 0; q < 3; ++q) fpp[q] = pp_s[q * Jp + fj];
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
    // prefetch this thread's xw (first pair) into shared memory before
    // waiting on h: an asynchronous copy, which neither the compiler nor the
    // assembler moves to the first use as they may a load into a register
    float* xsv = xs + (size_t)tid_c * G;
    if (tid_c < npairs) {
      const int pL = lens_s[fb];
      const bool pact = s < pL;
      const int pt = pact ? (reverse ? pL - 1 - s : s) : s;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (pact) {
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(xsv + g)),
                       "l"(p.xw + xw_index(p, d, pt, b0 + fb, g, j0 + fj))
                       : "memory");
        } else {
          xsv[g] = 0.0f;
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    bool timed_out = false;
    if constexpr (!GRID) {
      if (s >= 1) timed_out = !mbar_wait_bounded(smem_u32(&bars[cur]), (uint32_t)(((s - 1) >> 1) & 1), p.timeout_ns);
    }
    // rec = R . h_prev for all gate rows (GRU lbr=0: z and r rows only); the
    // grid kernel's h_prev is publication s + 1 (the prologue's is the first)
    if (!products(0, lbr0 ? 2 * Jp : G * Jp, hs + (size_t)cur * NBC * KP, p.hglob + (size_t)cur * p.D * p.N * KP,
                  ctr_h, (unsigned)(s + 1))) {
      alive = false;
      break;
    }
    if constexpr (!GRID) {
      if (__syncthreads_or(timed_out)) {
        if (tid == 0) atomicOr(p.status, 1);
        alive = false;
        break;
      }
    }

    if (lbr0) {
      // GRU, linear_before_reset = 0: z, r, then r (.) h_prev of every unit is exchanged
      for (int idx = tid_c; idx < npairs; idx += NTc) {
        const bool first = idx == tid_c;
        const int jl = first ? fj : idx % Jc, bl = first ? fb : idx / Jc;
        const int L = lens_s[bl];
        const bool active = s < L;
        const int t = active ? (reverse ? L - 1 - s : s) : s;
        float xz, xr;
        if (first) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          xz = xsv[0];
          xr = xsv[1];
        } else {
          xz = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, 0, j0 + jl)) : 0.0f;
          xr = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, 1, j0 + jl)) : 0.0f;
        }
        const float hp = hown[bl * J + jl];
        const float wz = first ? fwb[0] : wb_s[0 * Jp + jl], rz = first ? frb[0] : rb_s[0 * Jp + jl];
        const float wr = first ? fwb[1] : wb_s[1 * Jp + jl], rr = first ? frb[1] : rb_s[1 * Jp + jl];
        const float pz = ((xz + gs[(size_t)(0 * Jp + jl) * nb_ld + bl]) + wz) + rz;
        const float pr = ((xr + gs[(size_t)(1 * Jp + jl) * nb_ld + bl]) + wr) + rr;
        const float z = act<GEN, 0>(af, clip_pre(p.clip, pz));
        const float r = act<GEN, 0>(af, clip_pre(p.clip, pr));
        zs[bl * J + jl] = z;
        const float rh = r * hp;
        if constexpr (GRID) {
          p.rhglob[first ? fg0 : ((size_t)d * p.N + b0 + bl) * KP + j0 + jl] = rh;
        } else {
          rstage[bl * J + jl] = rh;
        }
      }
      if constexpr (GRID) {
        if (!producer) {
          asm volatile("fence.proxy.async.global;" ::: "memory");  // r.h is read by bulk copies
          asm volatile("bar.sync 1, %0;" ::"r"(NTc) : "memory");
          if (tid == 0) publish(ctr_rh);
        }
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
      if (!products(2 * Jp, Jp, rhs + (size_t)cur * NBC * KP, p.rhglob, ctr_rh, (unsigned)(s + 1))) {
        alive = false;
        break;
      }
      if constexpr (!GRID) __syncthreads();
    }

    // gate arithmetic and state update, one (unit, batch row) pair per thread
    // (grid kernel: the first pair's Y element is stored after the team
    // counter's release, which then waits only for the exchanged h)
    float y_first = 0.0f;
    size_t y_first_at = 0;
    for (int idx = tid_c; idx < npairs; idx += NTc) {
      const bool first = idx == tid_c;
      int jl, bl;
      size_t y0, g0;
      if (first) {
        jl = fj;
        bl = fb;
        y0 = fy0;
        g0 = fg0;
      } else {
        jl = idx % Jc;
        bl = idx / Jc;
        y0 = y_index(p, 0, d, b0 + bl, j0 + jl);
        g0 = ((size_t)d * p.N + b0 + bl) * KP + j0 + jl;
      }
      const int L = lens_s[bl];
      const bool active = s < L;
      const int t = active ? (reverse ? L - 1 - s : s) : s;
      // the pair's xw, biases and peepholes: the first pair's from the
      // prefetch and registers, any other's from memory
      float xv[G], wbv[G], rbv[G], ppv[3];
      if (first) {
        asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
        for (int g = 0; g < G; ++g) {
          xv[g] = xsv[g];
          wbv[g] = fwb[g];
          rbv[g] = frb[g];
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) ppv[q] = fpp[q];
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          xv[g] = active ? __ldcg(p.xw + xw_index(p, d, t, b0 + bl, g, j0 + jl)) : 0.0f;
          wbv[g] = wb_s[g * Jp + jl];
          rbv[g] = rb_s[g * Jp + jl];
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) ppv[q] = pp_s[q * Jp + jl];
      }
      const float hp = hown[bl * J + jl];
      float hn = hp;
      if (active) {
        float pre[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pre[g] = ((xv[g] + gs[(size_t)(g * Jp + jl) * nb_ld + bl]) + wbv[g]) + rbv[g];
        if constexpr (CELL == 0) {
          const float cp = cs[bl * J + jl];
          float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
          pi = has_p ? pi + ppv[0] * cp : pi;
          pf = has_p ? pf + ppv[2] * cp : pf;
          const float ig = act<GEN, 0>(af, clip_pre(p.clip, pi));
          const float fg = p.input_forget ? 1.0f - ig : act<GEN, 0>(af, clip_pre(p.clip, pf));
          const float cg = act<GEN, 1>(ag, clip_pre(p.clip, pc));
          const float cn = fg * cp + ig * cg;
          po = has_p ? po + ppv[1] * cn : po;
          const float og = act<GEN, 0>(af, clip_pre(p.clip, po));
          hn = og * act<GEN, 1>(ah, cn);
          cs[bl * J + jl] = cn;
        } else if constexpr (CELL == 1) {
          float z, ph;
          if (lbr0) {
            z = zs[bl * J + jl];
            ph = pre[2];  // ((xw_h + R_h.(r.h)) + Wb_h) + Rb_h
          } else {
            z = act<GEN, 0>(af, clip_pre(p.clip, pre[0]));
            const float r = act<GEN, 0>(af, clip_pre(p.clip, pre[1]));
            ph = (xv[2] + r * (gs[(size_t)(2 * Jp + jl) * nb_ld + bl] + rbv[2])) + wbv[2];
          }
          const float hc = act<GEN, 1>(ag, clip_pre(p.clip, ph));
          hn = (1.0f - z) * hc + z * hp;
        } else {
          hn = act<GEN, 1>(af, clip_pre(p.clip, pre[0]));
        }
      }
      hown[bl * J + jl] = hn;
      if (GRID && first) {
        y_first = active ? hn : 0.0f;
        y_first_at = y0 + (size_t)t * y_tstride;
      } else if (Y != nullptr) {
        store_elem<T>(Y + y0 + (size_t)t * y_tstride, active ? hn : 0.0f);
      }
      if constexpr (GRID) {
        p.hglob[(size_t)nxt * hbuf + g0] = hn;
      } else {
        stage[bl * J + jl] = hn;
      }
    }
    if constexpr (GRID) {
      // the computing threads are done with gs and have written h; the
      // staging warp is already waiting for the next step's h
      if (!producer) {
        asm volatile("fence.proxy.async.global;" ::: "memory");  // h is read by bulk copies
        asm volatile("bar.sync 1, %0;" ::"r"(NTc) : "memory");
        if (tid == 0 && s + 1 < p.T) publish(ctr_h);
        if (Y != nullptr && tid_c < npairs) store_elem<T>(Y + y_first_at, y_first);
      }
    } else if (s + 1 < p.T) {
      __syncthreads();
      push_slice(stage, hs + (size_t)nxt * NBC * KP, &bars[nxt]);
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
