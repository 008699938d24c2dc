// rk_step_tcs.cuh -- tensor-core recurrent step for small batches (at most 16
// rows per direction) of 16-bit layers (Half or bfloat16: the element type
// E) whose hidden units fit one cluster.  Instantiated by rk_step_tcs.cu
// (Half, and the entry point) and rk_step_tcs_bf16.cu (bfloat16).
//
// Same arithmetic as rk_step.cuh and rk_step_tc.cuh (web page "Recurrent
// layers", sections "How a layer runs" and "Arithmetic and determinism"):
// per step and gate row pre = ((xw + rec) + Wb) + Rb with rec = R_row .
// h_prev (h rounded to E for the product, state float32), then
// peepholes, clip, activation and state update (LSTM, RNN, GRU with
// linear_before_reset 0 or 1).
//
// With a small batch the product is turned around: the MMA's M = 128 rows
// are this CTA's gate rows (row g * 32 + u for gate g, unit u of its 32
// units; rows past G * 32 are zero) held in TMEM as the MMA's A operand for
// the whole layer, and its N = 16 columns are the direction's batch rows, so the
// exchanged operand is only 16 rows of h (2 KB per 64 k).  A team is one
// direction, one cluster of ceil(H / 32) CTAs.  Every CTA keeps the whole
// 16-bit operand, double-buffered, in its own shared memory in the layout
// the tensor cores read (H / 64 blocks of 16 rows x 64 k, 128-byte
// swizzled).  Per step:
//   1. one lane issues the H / 16 MMAs (kind::f16, M = 128, N = 16,
//      K = 16) on buffer s % 2 into one fp32 TMEM accumulator (lane = gate
//      row, column = batch row) once that buffer's byte-counting mbarrier
//      has completed;
//   2. warp g < G reads gate g's lanes (unit = lane) and stages them in
//      shared memory; every gate thread then takes one (unit, batch row)
//      pair (two when the batch exceeds 8) and does the gate arithmetic;
//   3. each warp packs its row's 32 new 16-bit h values into four 16-byte
//      chunks (shuffles) and pushes every chunk into buffer (s + 1) % 2 of
//      every CTA of the cluster with st.async, whose completion counts the
//      bytes on the receiver's mbarrier -- no global memory, no flags, no
//      copy back.
// A buffer is re-armed (expected bytes) before this CTA pushes the h that
// lets its peers produce the next value for it, and a peer can only write
// h_{s+2} into buffer s % 2 after it has every CTA's h_{s+1}, by which time
// every product that read h_s is complete.  GRU with linear_before_reset
// = 0 runs two rounds per step: the first product gives z and r, each warp
// pushes its 16-bit r (.) h_prev the same way into a second pair of buffers,
// and the second product gives R_h . (r (.) h).  Neither round needs all
// 128 rows of M, and an MMA costs the same whatever its rows, so the rounds
// stack k ranges into the rows instead: round 1 holds the z and r rows of
// the first and of the second half of k (4 x 32 rows) against the h rows of
// both halves (N = 32), round 2 the candidate rows of the four quarters of
// k (4 x 32 rows) against the r (.) h rows of the four quarters (N = 64);
// only the blocks of a k range times the same k range are used, and each
// gate sum is the sum of its ranges in increasing order.  H / 32 MMAs per
// step instead of H / 8.  The summation order is fixed (k in increasing
// 16-wide steps within a range, ranges in order), so runs are
// bit-identical.  Every wait is bounded; on expiry the kernel sets the
// status word, drains its MMAs, frees its TMEM and returns.
#pragma once
#include "rk_step_tc.cuh"

namespace rk {

namespace {

constexpr int XN = 16;         // MMA N: a direction's batch rows, padded
constexpr int XJ = 32;         // hidden units per CTA
constexpr int XPAIRS = 2;      // (unit, batch row) pairs per gate thread at most
constexpr int XBLK_B = XN * 128;   // bytes of one 64-k block of h
constexpr uint32_t XACC_COLS = 32;  // TMEM columns of the accumulator (one round: 16, rounded up)
// GRU with linear_before_reset = 0: k ranges stacked into the rows (F = 2
// ranges in round 1, 4 in round 2); TMEM columns of the round-1 accumulator
// (N = 32), the round-2 accumulator (N = 64) and the start of the gate rows
constexpr uint32_t XS_ACC1 = 0, XS_ACC2 = 64, XS_ROWS = 128;

// 64-k blocks per k range when the operand's k is cut into F ranges.
__host__ __device__ constexpr int tcs_blocks_per_range(int KB, int F) { return (KB + F - 1) / F; }

// TMEM columns the kernel allocates for hidden size H: the accumulators,
// then the CTA's gate rows as the MMA's A operand (lane = gate row, one
// column per two k), a power of two.  Stacked (GRU lbr 0): the z and r rows
// of two k halves, then the candidate rows of four k quarters.
__host__ __device__ inline uint32_t tcs_tmem_cols(int H, bool stacked) {
  const int KB = (H + SK - 1) / SK;
  if (stacked)
    return tmem_cols_for(XS_ROWS + (uint32_t)(tcs_blocks_per_range(KB, 2) + tcs_blocks_per_range(KB, 4)) * (SK / 2));
  return tmem_cols_for(XACC_COLS + (uint32_t)KB * (SK / 2));
}

// Bytes of one operand buffer: room for KB blocks of 16 rows, for 2 ranges
// of ceil(KB / 2) blocks of 32 rows and for 4 ranges of ceil(KB / 4)
// blocks of 64 rows alike (a multiple of 1 KB, the swizzle atom).
__host__ __device__ inline int tcs_buffer_bytes(int H) {
  const int KB = (H + SK - 1) / SK;
  return tcs_blocks_per_range(KB, 4) * 4 * XBLK_B;
}

// Byte offset of element (batch row b, k) in an operand buffer whose k is
// cut into F ranges of KBF = ceil(KB / F) blocks: block j of range q holds
// rows q * 16 + b of 64 consecutive k, 128-byte swizzled (F = 1: the plain
// layout, block kb = k / 64 of 16 rows).
__device__ __forceinline__ uint32_t tcs_operand_offset(int F, int KBF, int b, int k) {
  const int kb = k / SK, q = kb / KBF, j = kb - q * KBF;
  return (uint32_t)j * (uint32_t)(F * XBLK_B) + sw128_offset(q * XN + b, k % SK);
}

// 32 consecutive TMEM columns of this warp's 32 lanes from 32 registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// D (TMEM) += A (TMEM: lane = row of A, k packed two per column) . B^T
// (shared memory, descriptor), kind::f16, cta_group::1.
__device__ __forceinline__ void tc_mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Shared memory: [operands: [h, r (.) h][2 buffers][tcs_buffer_bytes]][staged
// products [4 gates][16 rows][32 units] floats][barriers][biases].  The gate
// rows live in TMEM.
struct XsSmem {
  size_t h, acc, bar, bias, total;
};
__host__ __device__ inline XsSmem xs_layout(int G, int H) {
  XsSmem L{};
  size_t o = 1024;  // room to align the dynamic base up to 1024 bytes
  L.h = o;    o += (size_t)2 * 2 * tcs_buffer_bytes(H);
  L.acc = o;  o += (size_t)4 * XJ * XN * 4;
  L.bar = o;  o += 256;
  L.bias = o; o += (size_t)2 * 4 * XJ * 4 + 3 * XJ * 4;
  L.total = o;
  (void)G;
  return L;
}

template <int CELL, bool GEN, bool PLAIN, bool LBR0, typename E>
__global__ void __launch_bounds__(STHREADS, 1) step_tcs_kernel(const StepParams p) {
  static_assert(!LBR0 || CELL == 1, "two rounds only for GRU with linear_before_reset = 0");
  constexpr int NRND = LBR0 ? 2 : 1;  // products per step
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  // accumulators (columns 0 .. 31), then the gate rows (A operand)
  const uint32_t kTmemCols = tcs_tmem_cols(p.H, LBR0);
  extern __shared__ unsigned char tsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  const XsSmem L = xs_layout(G, p.H);
  unsigned char* sH = base + (L.h - 1024);
  // staged products [g][b][u]: a gate thread's row b is warp-uniform and its
  // unit is the lane, so its reads are 32 consecutive floats (the layout
  // [g][u][b] had lanes 16 floats apart: 16-way bank conflicts)
  float* sAcc = reinterpret_cast<float*>(base + (L.acc - 1024));
  // operand arrived [round][buffer], drain, then per round: done, free, staged
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (L.bar - 1024));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
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
  const E* R = static_cast<const E*>(p.R);
  const E* Bias = static_cast<const E*>(p.Bias);
  const E* P = static_cast<const E*>(p.P);
  const E* h0 = static_cast<const E*>(p.h0);
  const E* c0 = static_cast<const E*>(p.c0);
  E* Y = static_cast<E*>(p.Y);

  // ---------------- prologue: biases, peepholes, operand buffers, barriers, TMEM
  for (int e = tid; e < G * XJ; e += blockDim.x) {
    const int g = e / XJ, u = e % XJ;
    const bool ok = j0 + u < H && Bias != nullptr;
    wb_s[e] = ok ? Elem<E>::to_f(Bias[(size_t)d * 2 * GH + (size_t)g * H + j0 + u]) : 0.0f;
    rb_s[e] = ok ? Elem<E>::to_f(Bias[(size_t)d * 2 * GH + GH + (size_t)g * H + j0 + u]) : 0.0f;
  }
  for (int e = tid; e < 3 * XJ; e += blockDim.x) {
    const int u = e / 3, g = e % 3;
    pp_s[e] = (CELL == 0 && !PLAIN && P != nullptr && j0 + u < H) ? Elem<E>::to_f(P[(size_t)d * 3 * H + (size_t)g * H + j0 + u]) : 0.0f;
  }
  // operand buffers: zero all (the k columns past the last CTA's units and
  // the rows past the batch belong to nobody; R is zero there too, but a
  // stale Inf or NaN times zero would not be), then h_0 into buffer 0
  const int KBB = tcs_buffer_bytes(H);  // bytes of one buffer
  // k ranges stacked into the rows of each operand (1: not stacked) and
  // 64-k blocks per range
  const int F0 = LBR0 ? 2 : 1, F1 = 4;
  const int KB0 = tcs_blocks_per_range(KB, F0), KB1 = tcs_blocks_per_range(KB, F1);
  for (int e = tid; e < 4 * KBB / 16; e += blockDim.x)
    reinterpret_cast<uint4*>(sH)[e] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  // byte offset of element (batch row b, k) of operand `which` in its buffer
  auto op_off = [&](int which, int b, int k) {
    return which == 0 ? tcs_operand_offset(F0, KB0, b, k) : tcs_operand_offset(F1, KB1, b, k);
  };
  auto sh_at = [&](int which, int buf, int b, int j) {
    return reinterpret_cast<E*>(sH + (size_t)(which * 2 + buf) * KBB + op_off(which, b, j));
  };
  for (int e = tid; e < N * H; e += blockDim.x) {
    const int b = e / H, j = e % H;
    *sh_at(0, 0, b, j) = Elem<E>::from_f(h0 != nullptr ? Elem<E>::to_f(h0[state_index(p, d, b, j)]) : 0.0f);
  }
  // bytes of one operand's arrival: C CTAs x N rows x 32 units x 2 bytes
  const uint32_t op_bytes = (uint32_t)C * (uint32_t)N * (uint32_t)(XJ * 2);
  auto full_bar = [&](int which, int buf) { return su32(&bars[which * 2 + buf]); };
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);  // operand [round][buffer] arrived
    mbar_init(smem_u32(&bars[4]), 1);                                // final MMA drain
    for (int rd = 0; rd < 2; ++rd) {
      uint64_t* b3 = bars + 5 + 3 * rd;
      mbar_init(smem_u32(&b3[0]), 1);  // accumulator complete (MMA commit)
      mbar_init(smem_u32(&b3[1]), 8);  // accumulator read (8 gate warps)
      mbar_init(smem_u32(&b3[2]), 8);  // products staged (8 gate warps)
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // h_0 was written locally: complete buffer 0's first phase; arm the
    // arrivals of h_1 and of r (.) h_0 before any CTA can push them
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(full_bar(0, 0)) : "memory");
    if (Tn > 1) mbar_arrive_expect_tx(full_bar(0, 1), op_bytes);
    if (LBR0 && Tn > 0) mbar_arrive_expect_tx(full_bar(1, 0), op_bytes);
  }
  // h_0 was written by ordinary stores; the tensor cores read it through
  // the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The gate rows (row g * 32 + u for gate g, unit u; zero past G * 32
  // rows, past H units and past H in k) go to TMEM once, as the MMA's A
  // operand: lane = row, column XACC_COLS + k / 2 holding k and k + 1.
  // From shared memory every MMA re-read its 4 KB of A there (the MMA's
  // cost tracks its operand bytes at these small N); from TMEM only the 512
  // bytes of h are read.  Warp w stores the rows of lane quarter w % 4 and
  // the 64-k blocks kb with kb % 2 == w / 4, one block (32 columns) at a time.
  // Stacked (GRU lbr 0): lane quarter Q holds from column XS_ROWS the z
  // (Q even) or r (Q odd) rows of k half Q / 2, ceil(KB / 2) blocks, and
  // after those the candidate rows of k quarter Q, ceil(KB / 4) blocks.
  if (warp < 8) {
    const int q = warp & 3;
    const bool r_vec = (reinterpret_cast<uintptr_t>(R) & 15) == 0;
    const uint32_t tlane = *tmem_slot + ((uint32_t)(32 * q) << 16);
    // 64 k of block kb of gate g's row of unit j0 + lane into 32 columns at col
    auto put_block = [&](int g, int kb, uint32_t col) {
      const int u = lane;
      const bool row_ok = g < G && j0 + u < H && kb < KB;
      const E* rrow = R + ((size_t)d * GH + (size_t)(row_ok ? g : 0) * H + (row_ok ? j0 + u : 0)) * H;
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = kb * SK + 8 * c;  // H is a multiple of 8: a chunk is wholly in or past H
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok && k < H) {
          if (r_vec) {
            w = __ldg(reinterpret_cast<const uint4*>(rrow + k));
          } else {
            __align__(16) E t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = rrow[k + i];
            w = *reinterpret_cast<const uint4*>(t8);
          }
        }
        v[4 * c + 0] = w.x;
        v[4 * c + 1] = w.y;
        v[4 * c + 2] = w.z;
        v[4 * c + 3] = w.w;
      }
      tmem_st32(tlane + col, v);
    };
    if constexpr (LBR0) {
      for (int j = warp >> 2; j < KB0; j += 2) put_block(q & 1, (q >> 1) * KB0 + j, XS_ROWS + (uint32_t)(j * (SK / 2)));
      for (int j = warp >> 2; j < KB1; j += 2)
        put_block(2, q * KB1 + j, XS_ROWS + (uint32_t)((KB0 + j) * (SK / 2)));
    } else {
      for (int kb = warp >> 2; kb < KB; kb += 2) put_block(q, kb, XACC_COLS + (uint32_t)(kb * (SK / 2)));
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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
      hreg[k] = h0 != nullptr ? Elem<E>::to_f(h0[si]) : 0.0f;
      creg[k] = (CELL == 0 && c0 != nullptr) ? Elem<E>::to_f(c0[si]) : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA's barriers are initialised and armed before any push (all
  // CTAs of a cluster run at once and reach this point)
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const uint32_t tmem_acc = *tmem_slot;

  const uint32_t bar_drain = su32(&bars[4]);
  // round rd's barriers: done, free, staged
  auto rbar = [&](int rd, int i) { return su32(&bars[5 + 3 * rd + i]); };
  // push this warp's batch row b of operand `which` (lane = unit, value v)
  // into buffer buf of every CTA: lanes 8c .. 8c + 7 form the 16-byte
  // chunk c of the row, lane l sends chunk l % 4 to CTAs l / 4, l / 4 + 8
  auto push_row = [&](int which, int buf, int b, float v) {
    const E e = Elem<E>::from_f(v);
    const uint32_t hv = (uint32_t)(*reinterpret_cast<const unsigned short*>(&e));
    const int c = lane & 3;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __shfl_sync(0xffffffffu, hv, 8 * c + 2 * i);
      const uint32_t hi = __shfl_sync(0xffffffffu, hv, 8 * c + 2 * i + 1);
      w[i] = lo | (hi << 16);
    }
    const int k = j0 + 8 * c;  // first unit of the chunk (the 8 units lie in one 64-k block)
    const uint32_t dst = su32(sH) + (uint32_t)((which * 2 + buf) * KBB) + op_off(which, b, k);
    const uint32_t bar = full_bar(which, buf);
    const float4 x = make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]), __uint_as_float(w[3]));
    for (int q = lane >> 2; q < C; q += 8) st_async_v4(map_to_rank(dst, (uint32_t)q), x, map_to_rank(bar, (uint32_t)q));
  };

  const size_t xw_tstride = p.layout == 0 ? (size_t)N * GH : GH;
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;

  if (warp == 9) {
    // ---------------- MMA lane: acc_rd[128 gate rows x 16 batch] = R_rows . operand^T
    // (stacked: acc_rd[128 rows of F k ranges x 16 F rows of the same F ranges])
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(XN) | Elem<E>::kMmaAB;
      const uint32_t idesc_st[2] = {idesc_f16(XN * 2) | Elem<E>::kMmaAB, idesc_f16(XN * 4) | Elem<E>::kMmaAB};
      const uint32_t ta0 = tmem_acc + XACC_COLS;  // the gate rows: 8 columns per 16 k
      constexpr uint64_t kK16 = 32 >> 4;
      bool ok = true;
      for (int s = 0; s < Tn && ok; ++s) {
        for (int rd = 0; rd < NRND; ++rd) {
          // operand rd of step s (buffer s % 2, its (s / 2)-th arrival)
          if (abort_flag || !bar_wait(full_bar(rd, s & 1), (uint32_t)((s >> 1) & 1), p.timeout_ns)) {
            ok = false;
            break;
          }
          // the peers' st.async writes, acquired above, are read by the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          // the gate warps must have read this accumulator of the previous step
          if (s > 0 && !bar_wait(rbar(rd, 1), (uint32_t)((s - 1) & 1), p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint64_t bd = desc_sw128(su32(sH) + (uint32_t)((rd * 2 + (s & 1)) * KBB));
          if constexpr (LBR0) {
            // round rd: F ranges of KBF blocks; block j of every range in one
            // MMA per 16 k (rows of range q times operand rows of range q
            // are the products used)
            const int F = rd == 0 ? F0 : F1, KBF = rd == 0 ? KB0 : KB1;
            const uint32_t tacc = tmem_acc + (rd == 0 ? XS_ACC1 : XS_ACC2);
            const uint32_t idn = idesc_st[rd];
            uint32_t ta = tmem_acc + XS_ROWS + (uint32_t)(rd == 0 ? 0 : KB0 * (SK / 2));
            const uint64_t bstep = (uint64_t)(F * XBLK_B) >> 4;
            for (int j = 0; j < KBF; ++j, ta += SK / 2, bd += bstep) {
              tc_mma_ts(tacc, ta, bd, idn, j != 0 ? 1u : 0u);
              tc_mma_ts(tacc, ta + 8, bd + kK16, idn, 1u);
              tc_mma_ts(tacc, ta + 16, bd + 2 * kK16, idn, 1u);
              tc_mma_ts(tacc, ta + 24, bd + 3 * kK16, idn, 1u);
            }
          } else {
            const uint32_t tacc = tmem_acc + (uint32_t)(rd * XN);
            uint32_t ta = ta0;
            for (int kb = 0; kb < KB; ++kb, ta += SK / 2, bd += XBLK_B >> 4) {
              tc_mma_ts(tacc, ta, bd, idesc, kb != 0 ? 1u : 0u);
              tc_mma_ts(tacc, ta + 8, bd + kK16, idesc, 1u);
              tc_mma_ts(tacc, ta + 16, bd + 2 * kK16, idesc, 1u);
              tc_mma_ts(tacc, ta + 24, bd + 3 * kK16, idesc, 1u);
            }
          }
          tc_commit(rbar(rd, 0));  // accumulator rd of step s complete
        }
      }
      if (!ok) {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
      // drain: every MMA this CTA issued completes before TMEM is freed
      tc_commit(bar_drain);
      bar_wait(bar_drain, 0u, p.timeout_ns);
    }
  } else if (gate_warp) {
    // ---------------- gate warps (warp 8 has no role)
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
    // wait for accumulator rd of step s, stage gates [g0, g1) of it (warp g
    // holds gate g of the 32 units, lane = unit) and make them visible to
    // every gate warp.  Stacked (GRU lbr 0): warp Q < 4 stages the sums of
    // its lane quarter over its own k range (round 1: gate Q % 2, half
    // Q / 2; round 2: the candidate gate, quarter Q) into slot Q.
    auto stage = [&](int rd, int s, int g0, int g1) -> bool {
      if (abort_flag || !bar_wait(rbar(rd, 0), (uint32_t)(s & 1), p.timeout_ns)) return false;
      tc_fence_after();
      if (LBR0 ? warp < 4 : (warp >= g0 && warp < g1)) {
        uint32_t col = (uint32_t)(rd * XN);
        if constexpr (LBR0) col = rd == 0 ? XS_ACC1 + (uint32_t)((warp >> 1) * XN) : XS_ACC2 + (uint32_t)(warp * XN);
        uint32_t v[XN];
        tmem_ld<XN>(tmem_acc + ((uint32_t)(warp * 32) << 16) + col, v);
#pragma unroll
        for (int b = 0; b < XN; ++b) sAcc[((size_t)warp * XN + b) * XJ + lane] = __uint_as_float(v[b]);
      }
      // the accumulator may be overwritten by the next step's product
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(rbar(rd, 1)) : "memory");
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(rbar(rd, 2)) : "memory");
      }
      return bar_wait(rbar(rd, 2), (uint32_t)(s & 1), p.timeout_ns);
    };
    float zr[XPAIRS][2];  // GRU linear_before_reset = 0: z and r between the rounds
    load_xw(0);
    bool ok = true;
    for (int s = 0; s < Tn; ++s) {
      if constexpr (LBR0) {
        // round 0: z and r; push r (.) h_prev
        if (!stage(0, s, 0, 2)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < XPAIRS; ++k) {
          if (!pv[k]) continue;  // the same for the whole warp
          const int b = (tid + 256 * k) >> 5;
          float pre[2];
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            // the two k halves of gate g's sum, in order
            const float rec = sAcc[((size_t)g * XN + b) * XJ + pu] + sAcc[((size_t)(g + 2) * XN + b) * XJ + pu];
            pre[g] = ((xv[k][g] + rec) + wb_s[g * XJ + pu]) + rb_s[g * XJ + pu];
          }
          zr[k][0] = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[0]));
          zr[k][1] = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[1]));
          push_row(1, s & 1, b, pj < H ? zr[k][1] * hreg[k] : 0.0f);
        }
      }
      // the last (or only) round: the remaining gate arithmetic
      constexpr int RL = NRND - 1;
      if (!stage(RL, s, LBR0 ? 2 : 0, G)) {
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
          if constexpr (LBR0) {
            // the candidate's sum: its four k quarters, in order
            const float* q0 = sAcc + (size_t)b * XJ + pu;
            rec[g] = g < 2 ? 0.0f : ((q0[0] + q0[XN * XJ]) + q0[2 * XN * XJ]) + q0[3 * XN * XJ];
          } else {
            rec[g] = sAcc[((size_t)g * XN + b) * XJ + pu];
          }
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
          float z, hc;
          if constexpr (LBR0) {
            // h~ = g(((xw_h + R_h . (r (.) h_prev)) + Wb_h) + Rb_h)
            z = zr[k][0];
            hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, pre[2]));
          } else {
            // linear_before_reset = 1: h~ = g((xw_h + r*(rec_h + Rb_h)) + Wb_h)
            z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[0]));
            const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[1]));
            const float ph = (xv[k][2] + r * (rec[2] + rb_s[2 * XJ + pu])) + wb_s[2 * XJ + pu];
            hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ph));
          }
          if (active) hn = (1.0f - z) * hc + z * hreg[k];
        } else {
          if (active) hn = act<GEN, 1>(p, d * A + 0, clip_pre(clip, pre[0]));
        }
        if (pj < H) hreg[k] = hn;
        if (Y != nullptr && pj < H) Y[y_index(p, t, d, b, pj)] = Elem<E>::from_f(active ? hn : 0.0f);
      }
      if (s + 1 < Tn) {
        // arm the arrivals this push lets the peers send: h_{s+2} into
        // buffer s % 2 (its h_s phase completed before this step's product)
        // and r (.) h_{s+1} into the second operand's buffer (s + 1) % 2
        if (tid == 0) {
          if (s + 2 < Tn) mbar_arrive_expect_tx(full_bar(0, s & 1), op_bytes);
          if (LBR0) mbar_arrive_expect_tx(full_bar(1, (s + 1) & 1), op_bytes);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < XPAIRS; ++k)
          if (pv[k]) push_row(0, (s + 1) & 1, (tid + 256 * k) >> 5, pj < H ? hreg[k] : 0.0f);
      }
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
          for (int t = Tn; t < S; ++t) Y[y_index(p, t, d, b, pj)] = Elem<E>::from_f(0.0f);
        const bool zero = S > 0 && lenv[k] == 0;
        const size_t si = state_index(p, d, b, pj);
        if (p.Yh != nullptr) static_cast<E*>(p.Yh)[si] = Elem<E>::from_f(zero ? 0.0f : hreg[k]);
        if (CELL == 0 && p.Yc != nullptr) static_cast<E*>(p.Yc)[si] = Elem<E>::from_f(zero ? 0.0f : creg[k]);
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

template <int CELL, bool GEN, bool PLAIN, bool LBR0, typename E>
cudaError_t step_tcs_launch(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident) {
  auto kern = step_tcs_kernel<CELL, GEN, PLAIN, LBR0, E>;
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
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CELL, bool LBR0, typename E>
cudaError_t step_tcs_cell(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q) {
  const bool plain = !(p.clip > 0.0f) && p.P == nullptr && !p.input_forget;
  if (p.generic_acts)
    return plain ? step_tcs_launch<CELL, true, true, LBR0, E>(p, plan, s, q)
                 : step_tcs_launch<CELL, true, false, LBR0, E>(p, plan, s, q);
  return plain ? step_tcs_launch<CELL, false, true, LBR0, E>(p, plan, s, q)
               : step_tcs_launch<CELL, false, false, LBR0, E>(p, plan, s, q);
}

template <typename E>
cudaError_t step_tcs_cells(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident) {
  switch (p.cell) {
    case 0: return step_tcs_cell<0, false, E>(p, plan, s, resident);
    case 1: return p.lbr ? step_tcs_cell<1, false, E>(p, plan, s, resident) : step_tcs_cell<1, true, E>(p, plan, s, resident);
    default: return step_tcs_cell<2, false, E>(p, plan, s, resident);
  }
}

}  // namespace

// bfloat16 layers (rk_step_tcs_bf16.cu)
cudaError_t step_tcs_bf16(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident);

}  // namespace rk
