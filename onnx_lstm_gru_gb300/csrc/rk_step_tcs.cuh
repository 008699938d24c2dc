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
// the whole layer, and its N = 16 columns are the direction's batch rows,
// so the exchanged operand is only 16 rows of h (2 KB per 64 k).  A team is
// one direction, one cluster of ceil(H / 32) CTAs.  Every CTA keeps the
// whole 16-bit operand, double-buffered, in its own shared memory in the
// layout the tensor cores read (128-byte swizzled rows of 64 k).  Per step:
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
// every product that read h_s is complete.
//
// GRU with linear_before_reset = 0 needs r before it can exchange
// r (.) h_prev, and the candidate's product only after that exchange, so
// two products lie on each step's chain.  An MMA costs about the same
// whatever its rows, so there the gates are multiplied one at a time with
// k quarters stacked into the rows ("stacked"): the 32 rows of gate g for
// k quarter q sit in TMEM lane quarter q, and the operand's rows for
// quarter q are rows 16 q + b of a 64-row tile; one MMA per 16 k of a
// quarter's blocks multiplies all four quarters at once into gate g's
// accumulator (128 lanes x 64 columns), of which the blocks quarter q times
// quarter q (lanes 32 q .., columns 16 q ..) are used, and a gate's sum is
// its four quarters added in order.  r is multiplied first (H / 64 MMAs),
// each warp pushes its 16-bit r (.) h_prev into a second pair of buffers
// while z is multiplied, and the candidate's rows are multiplied against
// that operand: 2 H / 64 MMAs on the chain instead of 2 H / 16.  An RNN's
// one gate fills only 32 of the 128 rows, so it is stacked the same way:
// H / 64 MMAs per step instead of H / 16.  (For LSTM and GRU with
// linear_before_reset = 1 all gates are on the chain at once, and the plain
// single product was measured faster than three stacked ones.)  The summation
// order is fixed (k in increasing 16-wide steps, quarters in order), so
// runs are bit-identical.  Every wait is bounded; on expiry the kernel sets
// the status word, drains its MMAs, frees its TMEM and returns.
#pragma once
#include "rk_step_tc.cuh"

namespace rk {

namespace {

constexpr int XN = 16;         // MMA N per k range: a direction's batch rows, padded
constexpr int XJ = 32;         // hidden units per CTA
constexpr int XQ = 4;          // k quarters stacked into the MMA rows (GRU lbr 0, RNN)
constexpr int XPAIRS = 2;      // (unit, batch row) pairs per gate thread at most
constexpr int XBLK_B = XN * 128;        // bytes of one 64-k block of the plain operand (16 rows)
constexpr int XBLKQ_B = XQ * XBLK_B;    // bytes of one 64-k block of the stacked operand (64 rows)
constexpr uint32_t XACC_COLS = 32;      // plain: TMEM columns of the accumulator (16, rounded up)
constexpr uint32_t XACC = XQ * XN;      // stacked: TMEM columns of one gate's accumulator (N = 64)

// 64-k blocks per k quarter.
__host__ __device__ constexpr int tcs_quarter_blocks(int H) { return ((H + SK - 1) / SK + XQ - 1) / XQ; }

// TMEM columns the kernel allocates for hidden size H and G gates, a power
// of two.  Plain: the accumulator, then the gate rows (lane = row g * 32 + u,
// one column per two k).  Stacked: G accumulators of 64 columns, then gate
// g's rows (lane = 32 q + u for k quarter q).
__host__ __device__ inline uint32_t tcs_tmem_cols(int H, int G, bool stacked) {
  if (stacked) return tmem_cols_for((uint32_t)G * (XACC + (uint32_t)tcs_quarter_blocks(H) * (SK / 2)));
  return tmem_cols_for(XACC_COLS + (uint32_t)((H + SK - 1) / SK) * (SK / 2));
}

// Bytes of one operand buffer, room for either layout (a multiple of 8 KB).
__host__ __device__ inline int tcs_buffer_bytes(int H) { return tcs_quarter_blocks(H) * XBLKQ_B; }

// Byte offset of element (batch row b, k) in an operand buffer, 128-byte
// swizzled rows of 64 k.  Plain: block kb = k / 64 holds rows b.  Stacked:
// block j of quarter q (KBQ blocks per quarter) holds rows 16 q + b.
__device__ __forceinline__ uint32_t tcs_operand_offset(bool stacked, int KBQ, int b, int k) {
  const int kb = k / SK;
  if (!stacked) return (uint32_t)kb * (uint32_t)XBLK_B + sw128_offset(b, k % SK);
  const int q = kb / KBQ, j = kb - q * KBQ;
  return (uint32_t)j * (uint32_t)XBLKQ_B + sw128_offset(q * XN + b, k % SK);
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
// quarter sums [4 gates][4 quarters][16 rows][32 units] floats][barriers]
// [biases].  The gate rows live in TMEM.
struct XsSmem {
  size_t h, acc, bar, bias, total;
};
__host__ __device__ inline XsSmem xs_layout(int G, int H) {
  XsSmem L{};
  size_t o = 1024;  // room to align the dynamic base up to 1024 bytes
  L.h = o;    o += (size_t)2 * 2 * tcs_buffer_bytes(H);
  L.acc = o;  o += (size_t)4 * XQ * XJ * XN * 4;
  L.bar = o;  o += 256;
  L.bias = o; o += (size_t)2 * 4 * XJ * 4 + 3 * XJ * 4;
  L.total = o;
  (void)G;
  return L;
}

template <int CELL, bool GEN, bool PLAIN, bool LBR0, typename E>
__global__ void __launch_bounds__(STHREADS, 1) step_tcs_kernel(const StepParams p) {
  static_assert(!LBR0 || CELL == 1, "r (.) h exchange only for GRU with linear_before_reset = 0");
  // k quarters stacked into the MMA rows: GRU lbr 0 (three gates, one at a
  // time) and RNN (its one gate fills only 32 rows)
  constexpr bool STK = LBR0 || CELL == 2;
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  // accumulators, then the gate rows (A operand): see tcs_tmem_cols
  const uint32_t kTmemCols = tcs_tmem_cols(p.H, G, STK);
  extern __shared__ unsigned char tsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  const XsSmem L = xs_layout(G, p.H);
  unsigned char* sH = base + (L.h - 1024);
  // staged quarter sums [g][q][b][u]: a gate thread's row b is warp-uniform
  // and its unit is the lane, so its reads are 32 consecutive floats (the
  // layout [g][u][b] had lanes 16 floats apart: 16-way bank conflicts)
  float* sAcc = reinterpret_cast<float*>(base + (L.acc - 1024));
  // operand arrived [operand][buffer], drain, then per gate: done, free, staged
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (L.bar - 1024));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
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
  const int KBQ = tcs_quarter_blocks(H);  // 64-k blocks per k quarter
  for (int e = tid; e < 4 * KBB / 16; e += blockDim.x)
    reinterpret_cast<uint4*>(sH)[e] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  auto sh_at = [&](int which, int buf, int b, int j) {
    return reinterpret_cast<E*>(sH + (size_t)(which * 2 + buf) * KBB + tcs_operand_offset(STK, KBQ, b, j));
  };
  for (int e = tid; e < N * H; e += blockDim.x) {
    const int b = e / H, j = e % H;
    *sh_at(0, 0, b, j) = Elem<E>::from_f(h0 != nullptr ? Elem<E>::to_f(h0[state_index(p, d, b, j)]) : 0.0f);
  }
  // bytes of one operand's arrival: C CTAs x N rows x 32 units x 2 bytes
  const uint32_t op_bytes = (uint32_t)C * (uint32_t)N * (uint32_t)(XJ * 2);
  auto full_bar = [&](int which, int buf) { return su32(&bars[which * 2 + buf]); };
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);  // operand [h, r (.) h][buffer] arrived
    mbar_init(smem_u32(&bars[4]), 1);                                // final MMA drain
    for (int a = 0; a < G; ++a) {
      uint64_t* b3 = bars + 5 + 3 * a;
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
  // The gate rows go to TMEM once, as the MMA's A operand (zero past H
  // units, past G gates and past H in k), one column per two k.  From
  // shared memory every MMA re-read its 4 KB of A there (the MMA's cost
  // tracks its operand bytes at these small N); from TMEM only the operand
  // is read.  Plain: row g * 32 + u in lane quarter g from column 32, warp w
  // storing lane quarter w % 4 and the blocks kb with kb % 2 == w / 4.
  // Stacked: gate g's rows of k quarter q in lanes 32 q + u from column
  // G * 64 + g * KBQ * 32, warp w storing the blocks (g, j) with
  // (g * KBQ + j) % 2 == w / 4; one block (32 columns) at a time.
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
    if constexpr (STK) {
      for (int i = warp >> 2; i < G * KBQ; i += 2) {
        const int g = i / KBQ, j = i % KBQ;
        put_block(g, q * KBQ + j, (uint32_t)(G * XACC) + (uint32_t)(i * (SK / 2)));
      }
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
  // gate g's barriers: accumulator complete (MMA commit), read (8 gate
  // warps), quarter sums staged (8 gate warps)
  auto gbar = [&](int g, int i) { return su32(&bars[5 + 3 * g + i]); };
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
    const uint32_t dst = su32(sH) + (uint32_t)((which * 2 + buf) * KBB) + tcs_operand_offset(STK, KBQ, b, k);
    const uint32_t bar = full_bar(which, buf);
    const float4 x = make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]), __uint_as_float(w[3]));
    for (int q = lane >> 2; q < C; q += 8) st_async_v4(map_to_rank(dst, (uint32_t)q), x, map_to_rank(bar, (uint32_t)q));
  };

  const size_t xw_tstride = p.layout == 0 ? (size_t)N * GH : GH;
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;

  if (warp == 9) {
    // ---------------- MMA lane.  Stacked: per gate g, acc_g[128 rows of 4 k
    // quarters x 64 operand rows of the same 4 quarters] = gate g's rows .
    // operand^T
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(STK ? (int)XACC : XN) | Elem<E>::kMmaAB;
      constexpr uint64_t kK16 = 32 >> 4;
      constexpr uint64_t kBlk = (uint64_t)(STK ? XBLKQ_B : XBLK_B) >> 4;
      bool ok = true;
      for (int s = 0; s < Tn && ok; ++s) {
        if constexpr (!STK) {
          // plain: acc[128 gate rows x 16 batch rows] = R_rows . h^T over all of k
          if (abort_flag || !bar_wait(full_bar(0, s & 1), (uint32_t)((s >> 1) & 1), p.timeout_ns)) {
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          if (s > 0 && !bar_wait(gbar(0, 1), (uint32_t)((s - 1) & 1), p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t ta = tmem_acc + XACC_COLS;
          uint64_t bd = desc_sw128(su32(sH) + (uint32_t)((s & 1) * KBB));
          for (int kb = 0; kb < KB; ++kb, ta += SK / 2, bd += kBlk) {
            tc_mma_ts(tmem_acc, ta, bd, idesc, kb != 0 ? 1u : 0u);
            tc_mma_ts(tmem_acc, ta + 8, bd + kK16, idesc, 1u);
            tc_mma_ts(tmem_acc, ta + 16, bd + 2 * kK16, idesc, 1u);
            tc_mma_ts(tmem_acc, ta + 24, bd + 3 * kK16, idesc, 1u);
          }
          tc_commit(gbar(0, 0));  // accumulator of step s complete
        } else {
          // stacked.  GRU lbr 0: r first (its r (.) h goes out while z is
          // multiplied), then z, then the candidate against r (.) h.  RNN:
          // its one gate against h.
          for (int i = 0; i < G; ++i) {
            const int g = LBR0 ? (i == 0 ? 1 : (i == 1 ? 0 : 2)) : i;
            const int which = (LBR0 && g == 2) ? 1 : 0;
            if (i == 0 || which == 1) {
              // operand `which` of step s (buffer s % 2, its (s / 2)-th arrival)
              if (abort_flag || !bar_wait(full_bar(which, s & 1), (uint32_t)((s >> 1) & 1), p.timeout_ns)) {
                ok = false;
                break;
              }
              // the peers' st.async writes, acquired above, are read by the async proxy
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            // the gate warps must have read this accumulator of the previous step
            if (s > 0 && !bar_wait(gbar(g, 1), (uint32_t)((s - 1) & 1), p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_acc + (uint32_t)g * XACC;
            uint32_t ta = tmem_acc + (uint32_t)(G * XACC) + (uint32_t)(g * KBQ * (SK / 2));
            uint64_t bd = desc_sw128(su32(sH) + (uint32_t)((which * 2 + (s & 1)) * KBB));
            for (int j = 0; j < KBQ; ++j, ta += SK / 2, bd += kBlk) {
              tc_mma_ts(tacc, ta, bd, idesc, j != 0 ? 1u : 0u);
              tc_mma_ts(tacc, ta + 8, bd + kK16, idesc, 1u);
              tc_mma_ts(tacc, ta + 16, bd + 2 * kK16, idesc, 1u);
              tc_mma_ts(tacc, ta + 24, bd + 3 * kK16, idesc, 1u);
            }
            tc_commit(gbar(g, 0));  // accumulator g of step s complete
          }
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
    // Stacked: wait for gate g's accumulator of step s; the four warps of
    // lane group g % 2 (warp w: lane quarter w % 4, i.e. k quarter q) stage
    // the sums of their quarter (unit = lane) in shared memory.  Plain (g =
    // 0, the one accumulator): warp w < G stages gate w (its lane quarter).
    // Every gate warp then marks the accumulator read and the sums staged.
    auto stage = [&](int g, int s) -> bool {
      if (abort_flag || !bar_wait(gbar(g, 0), (uint32_t)(s & 1), p.timeout_ns)) return false;
      tc_fence_after();
      if (STK ? (warp >> 2) == (g & 1) : warp < G) {
        const int q = warp & 3;
        const int sg = STK ? g : warp, sq = STK ? q : 0;  // the slot: gate, quarter
        uint32_t v[XN];
        tmem_ld<XN>(tmem_acc + ((uint32_t)(q * 32) << 16) + (STK ? (uint32_t)g * XACC + (uint32_t)(q * XN) : 0u), v);
        float* dst = sAcc + (size_t)(sg * XQ + sq) * XN * XJ + lane;
#pragma unroll
        for (int b = 0; b < XN; ++b) dst[(size_t)b * XJ] = __uint_as_float(v[b]);
      }
      // the accumulator may be overwritten by the next step's product
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gbar(g, 1)) : "memory");
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gbar(g, 2)) : "memory");
      }
      return true;
    };
    auto staged = [&](int g, int s) { return bar_wait(gbar(g, 2), (uint32_t)(s & 1), p.timeout_ns); };
    // gate g's sum for batch row b and this thread's unit (stacked: its four
    // k quarters added in order)
    auto gsum = [&](int g, int b) {
      const float* q0 = sAcc + ((size_t)g * XQ * XN + b) * XJ + pu;
      if constexpr (!STK) return q0[0];
      return ((q0[0] + q0[XN * XJ]) + q0[2 * XN * XJ]) + q0[3 * XN * XJ];
    };
    load_xw(0);
    bool ok = true;
    for (int s = 0; s < Tn; ++s) {
      if constexpr (LBR0) {
        // r first; push r (.) h_prev; then z and the candidate (against r (.) h)
        if (!stage(1, s) || !staged(1, s)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < XPAIRS; ++k) {
          if (!pv[k]) continue;  // the same for the whole warp
          const int b = (tid + 256 * k) >> 5;
          const float pr = ((xv[k][1] + gsum(1, b)) + wb_s[1 * XJ + pu]) + rb_s[1 * XJ + pu];
          const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pr));
          push_row(1, s & 1, b, pj < H ? r * hreg[k] : 0.0f);
        }
        if (!stage(0, s) || !stage(2, s) || !staged(0, s) || !staged(2, s)) {
          ok = false;
          break;
        }
      } else if (!stage(0, s) || !staged(0, s)) {
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
          rec[g] = (LBR0 && g == 1) ? 0.0f : gsum(g, b);  // r was done above
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
            z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[0]));
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
