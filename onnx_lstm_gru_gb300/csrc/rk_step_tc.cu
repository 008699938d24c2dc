// rk_step_tc.cu -- persistent recurrent-step kernel on the tcgen05 tensor
// cores, for Half layers whose batch makes R . h a dense product.
//
// What it computes is the same as rk_step.cuh (web page "Recurrent layers",
// sections "How a layer runs" and "Arithmetic and determinism"): per step and
// gate row pre = ((xw + rec) + Wb) + Rb with rec = R_row . h_prev, then
// peepholes, clip, activation and state update (LSTM, RNN, GRU with
// linear_before_reset = 1).  The state (h, c) stays float32 in registers;
// the product's h operand is the state rounded to Half, so R (Half, exact)
// times that operand is exact in float32 and summed in float32.
//
// Layout: a team per (direction, group of up to 128 batch rows); a team is
// ceil(H / 16) CTAs, each owning 16 hidden units, all CTAs of the launch
// co-resident (cooperative launch).  A CTA keeps its 16 units' G rows of R in
// shared memory, unit-major (row u*G + g), in the 128-byte swizzled K-major
// layout the tensor cores read.  Per step:
//   1. one lane streams h_t through an 8-stage ring, one contiguous bulk copy
//      per 64-wide k block: the Half copy of h is kept in global memory
//      already in the swizzled K-major layout, one block of (team batch rows
//      rounded up to 64) x 64 k per k block, written 16 bytes at a time by the
//      gate threads;
//   2. one lane issues tcgen05.mma kind::f16 with M = 128 (batch rows),
//      N = 16 G (the CTA's gate rows), K = 16 per instruction, 64-wide k
//      block kb into fp32 TMEM accumulator kb % 4 (lane = batch row, column =
//      gate row): small-N MMAs into one accumulator would each wait for the
//      previous one; then commits to an mbarrier;
//   3. eight warps read the accumulator with tcgen05.ld: thread (warp w,
//      lane l) takes batch row 32 (w % 4) + l and 8 units (half w / 4), does
//      the gate arithmetic with its units' c and h in registers and the next
//      step's xw prefetched, writes Y and the Half copy of the new h;
//   4. the team passes a counter barrier with a bounded, timed wait.
// The summation order is fixed by the shape (tensor-core k blocks of 16 in
// increasing k within each accumulator, then ((a0 + a1) + (a2 + a3))), so
// runs are bit-identical.  Every wait is bounded; on
// expiry the kernel sets the status word, drains its copies and MMAs, frees
// its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "rk_step.cuh"

namespace rk {

namespace {

constexpr int SB = 128;          // batch rows per team (MMA M)
constexpr int SK = 64;           // k per ring stage (one 128-byte swizzle atom of Half)
constexpr int SRING = 64 * 1024; // bytes of the h ring: 8 stages of 64 rows or 4 of 128
constexpr int SMAXST = 8;
constexpr int SJ = 16;           // hidden units per CTA
constexpr int STHREADS = 320;    // 8 gate warps + producer warp + MMA warp

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(par)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_wait(uint32_t b, uint32_t par, long long timeout_ns) {
  if (bar_try(b, par)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (bar_try(b, par)) return true;
    if ((it & 15u) == 0 && (long long)(global_ns() - t0) > timeout_ns) return false;
  }
}
__device__ __forceinline__ void bar_expect(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16, A and B Half, D float32, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(SB >> 4) << 24);
}
// Byte offset of element (row r, k) of a K-major tile of 64-element rows in
// the 128-byte swizzled layout (16-byte chunks of a row XORed with r % 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  const int chunk = (k >> 3) ^ (r & 7);
  return (uint32_t)(r * 128 + chunk * 16 + (k & 7) * 2);
}
template <int NCOL>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[NCOL]);
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<24>(uint32_t taddr, uint32_t (&r)[24]) {
  uint32_t a[16], b[8];
  tmem_ld<16>(taddr, a);
  tmem_ld<8>(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = a[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[16 + i] = b[i];
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
  uint32_t a[16], b[16];
  tmem_ld<16>(taddr, a);
  tmem_ld<16>(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    r[i] = a[i];
    r[16 + i] = b[i];
  }
}

// Shared memory: [R slice: KB blocks of (16 G rows x 64 k) Half][ring: 4 x 16 KB][barriers]
struct TcSmem {
  size_t r, ring, bar, bias, total;
};
__host__ __device__ inline TcSmem tc_smem_layout(int G, int H) {
  TcSmem L{};
  const int KB = (H + SK - 1) / SK;
  const size_t rbytes = (size_t)KB * SJ * G * SK * 2;
  size_t o = 1024;  // room to align the dynamic base up to 1024 bytes
  L.r = o;    o += (rbytes + 1023) & ~(size_t)1023;
  // the MMA reads 128 rows (16 KB) of every stage; with 64-row stages the
  // last stage's upper half runs 8 KB past the ring, into this pad
  L.ring = o; o += (size_t)SRING + 8 * 1024;
  L.bar = o;  o += 256;
  L.bias = o; o += (size_t)2 * SJ * G * 4 + 3 * SJ * 4;
  L.total = o;
  return L;
}

// Half copy of the exchanged h, pre-arranged for the tensor cores: for every
// (buffer, direction, team, 64-wide k block) a contiguous block of box rows
// x 64 k in the 128-byte swizzled K-major layout, so one stage of the ring is
// one contiguous bulk copy.  Element (row, k) of a block sits at
// sw128_offset(row, k).
__device__ __forceinline__ size_t h16_block(const StepParams& p, int buf, int d, int team_in_dir, int kb, int KB,
                                            int box_rows) {
  return ((((size_t)buf * p.D + d) * p.teams_per_dir + team_in_dir) * KB + kb) * (size_t)box_rows * SK;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

template <int CELL, bool GEN, bool PLAIN>
__global__ void __launch_bounds__(STHREADS, 1) step_tc_kernel(const StepParams p, __half* __restrict__ h16) {
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  constexpr int NR = SJ * G;      // gate rows of this CTA (MMA N): 64, 48 or 16
  constexpr int UH = SJ / 2;      // units per gate thread
  constexpr int NCOL = UH * G;    // accumulator columns per gate thread
  extern __shared__ unsigned char tsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  const TcSmem L = tc_smem_layout(G, p.H);
  unsigned char* sR = base + (L.r - 1024);
  unsigned char* sRing = base + (L.ring - 1024);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (L.bar - 1024));  // full[8], empty[8], mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  float* wb_s = reinterpret_cast<float*>(base + (L.bias - 1024));
  float* rb_s = wb_s + NR;
  float* pp_s = rb_s + NR;
  __shared__ int flag_smem;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, N = p.N, S = p.S, Tn = p.T;
  const int C = p.team_ctas;
  const int team = blockIdx.x / C, rank = blockIdx.x % C;
  const int d = team / p.teams_per_dir;
  const int b0 = (team % p.teams_per_dir) * SB;
  const int nbt = min(SB, N - b0);
  const int j0 = rank * SJ;
  const int KB = (H + SK - 1) / SK;
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const size_t GH = (size_t)G * H;
  const __half* R = static_cast<const __half*>(p.R);
  const __half* Bias = static_cast<const __half*>(p.Bias);
  const __half* P = static_cast<const __half*>(p.P);
  const __half* h0 = static_cast<const __half*>(p.h0);
  const __half* c0 = static_cast<const __half*>(p.c0);
  __half* Y = static_cast<__half*>(p.Y);
  const int tin = team % p.teams_per_dir;      // team index within its direction
  // rows of h per ring stage: the team's batch rounded up to 64 (the MMA
  // still spans 128 rows; rows past the stage's are never read back)
  const int box_rows = p.nbc;                      // 64 or 128, set by the host
  const uint32_t stage_bytes = (uint32_t)box_rows * SK * 2;
  const int nstages = SRING / (int)stage_bytes;     // 8 or 4

  // ---------------- prologue: R slice (unit-major rows, swizzled), biases, barriers, TMEM
  for (size_t e = tid; e < (size_t)KB * NR * SK; e += blockDim.x) {
    const int kb = (int)(e / ((size_t)NR * SK));
    const int rem = (int)(e % ((size_t)NR * SK));
    const int r = rem / SK, kk = rem % SK;
    const int u = r / G, g = r % G, k = kb * SK + kk;
    __half v = __float2half(0.0f);
    if (j0 + u < H && k < H) v = R[((size_t)d * GH + (size_t)g * H + j0 + u) * H + k];
    *reinterpret_cast<__half*>(sR + (size_t)kb * NR * 128 + sw128_offset(r, kk)) = v;
  }
  for (int e = tid; e < NR; e += blockDim.x) {
    const int u = e / G, g = e % G;
    const bool ok = j0 + u < H && Bias != nullptr;
    wb_s[e] = ok ? __half2float(Bias[(size_t)d * 2 * GH + (size_t)g * H + j0 + u]) : 0.0f;
    rb_s[e] = ok ? __half2float(Bias[(size_t)d * 2 * GH + GH + (size_t)g * H + j0 + u]) : 0.0f;
  }
  for (int e = tid; e < 3 * SJ; e += blockDim.x) {
    const int u = e / 3, g = e % 3;
    pp_s[e] = (CELL == 0 && !PLAIN && P != nullptr && j0 + u < H) ? __half2float(P[(size_t)d * 3 * H + (size_t)g * H + j0 + u]) : 0.0f;
  }
  if (tid == 0) {
    for (int i = 0; i < SMAXST; ++i) {
      mbar_init(smem_u32(&bars[i]), 1);
      mbar_init(smem_u32(&bars[SMAXST + i]), 1);
    }
    mbar_init(smem_u32(&bars[2 * SMAXST]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // R was written by ordinary stores; the tensor cores read it through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  // four accumulators (k blocks kb % 4), so consecutive MMAs do not wait on
  // each other's results; columns 64 apart
  constexpr int NACC = 4;
  constexpr uint32_t kAccStride = 64;
  constexpr uint32_t kTmemCols = NACC * kAccStride;
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // gate threads: warps 0..7; batch row br = 32 (warp % 4) + lane, units [uh0, uh0 + 8)
  const bool gate_warp = warp < 8;
  const int q = warp & 3;
  const int uh0 = (warp >> 2) * UH;
  const int br = q * 32 + lane;
  const bool grow = gate_warp && br < nbt;
  const int bg = b0 + br;  // global batch row
  float hreg[UH], creg[UH];
  int len = Tn;
  if (grow) {
    if (p.lens != nullptr) {
      len = p.lens[bg];
      len = len < 0 ? 0 : (len > S ? S : len);
      len = len > Tn ? Tn : len;
    }
#pragma unroll
    for (int u = 0; u < UH; ++u) {
      const int j = j0 + uh0 + u;
      const size_t si = state_index(p, d, bg, j < H ? j : 0);
      hreg[u] = (j < H && h0 != nullptr) ? __half2float(h0[si]) : 0.0f;
      creg[u] = (CELL == 0 && j < H && c0 != nullptr) ? __half2float(c0[si]) : 0.0f;
      // h_0 into buffer 0 (units past H are zero: the k padding of the product)
      *reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(h16 + h16_block(p, 0, d, tin, j / SK, KB, box_rows)) +
                                 sw128_offset(br, j % SK)) = __float2half_rn(j < H ? hreg[u] : 0.0f);
    }
    // k columns past the last CTA's units (up to the 64-wide block) belong to
    // no CTA: zero them once in both buffers (R is zero there too, but a stale
    // Inf or NaN times zero would not be)
    if (rank == C - 1 && uh0 == 0) {
      for (int k = C * SJ; k < KB * SK; ++k)
        for (int buf = 0; buf < 2; ++buf)
          *reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(h16 + h16_block(p, buf, d, tin, k / SK, KB, box_rows)) +
                                     sw128_offset(br, k % SK)) = __float2half_rn(0.0f);
    }
  } else {
#pragma unroll
    for (int u = 0; u < UH; ++u) hreg[u] = creg[u] = 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_acc = *tmem_slot;

  unsigned nbar = 0;
  // h_0 copies were written by ordinary stores and are read by TMA (async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  bool alive = team_barrier(p.counters + team, (unsigned)C * (++nbar), p.timeout_ns, p.status, &flag_smem);

  // xw of this thread's units for step s: Xw[d][m(t, bg)][g*H + j]
  const size_t xw_tstride = p.layout == 0 ? (size_t)N * GH : GH;
  const float* xw_row = p.xw + xw_index(p, d, 0, grow ? bg : 0, 0, 0);
  // the 8 units of a gate are 32 contiguous bytes: two 16-byte loads when
  // they are aligned and all inside H
  const bool xw_vec = (j0 + uh0 + UH <= H) && (H % 4 == 0) && (reinterpret_cast<uintptr_t>(p.xw) % 16 == 0);
  auto load_xw = [&](int s, float (&x)[UH * G]) {
    const bool on = grow && s < len && s < Tn;
    const float* qx = xw_row + (size_t)(reverse ? len - 1 - s : s) * xw_tstride;
    if (on && xw_vec) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(qx + (size_t)g * H + j0 + uh0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(qx + (size_t)g * H + j0 + uh0 + 4));
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < UH; ++u) x[u * G + g] = v[u];
      }
    } else {
#pragma unroll
      for (int u = 0; u < UH; ++u)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int j = j0 + uh0 + u;
          x[u * G + g] = (on && j < H) ? __ldg(qx + (size_t)g * H + j) : 0.0f;
        }
    }
  };
  float xv[UH * G];
  load_xw(0, xv);
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;
  const size_t ystride = p.layout == 0 ? (size_t)p.D * N * H : (size_t)p.D * H;
  const uint32_t idesc = idesc_f16(NR);

  int stage = 0;       // ring position, shared by producer and MMA lanes
  uint32_t phase = 0;
  int armed[SMAXST];
  for (int i = 0; i < SMAXST; ++i) armed[i] = -1;

  for (int s = 0; s < Tn && alive; ++s) {
    const int cur = s & 1, nxt = cur ^ 1;
    if (warp == 8 && lane == 0) {
      // ---- producer: h_s rows [d*N + b0, +128) in 64-k blocks
      asm volatile("fence.proxy.async.global;" ::: "memory");
      int st = stage;
      uint32_t ph = phase;
      for (int kb = 0; kb < KB && !abort_flag; ++kb) {
        if (!bar_wait(su32(&bars[SMAXST + st]), ph ^ 1u, p.timeout_ns)) {
          abort_flag = 1;
          atomicOr(p.status, 1);
          break;
        }
        bar_expect(su32(&bars[st]), stage_bytes);
        bulk_load(su32(sRing + st * stage_bytes), h16 + h16_block(p, cur, d, tin, kb, KB, box_rows), stage_bytes,
                  su32(&bars[st]));
        armed[st] = (int)ph;
        if (++st == nstages) {
          st = 0;
          ph ^= 1u;
        }
      }
    } else if (warp == 9 && lane == 0) {
      // ---- MMA: acc[128 x NR] = h_s[128 x H] . R_slice[NR x H]^T
      int st = stage;
      uint32_t ph = phase;
      for (int kb = 0; kb < KB && !abort_flag; ++kb) {
        if (!bar_wait(su32(&bars[st]), ph, p.timeout_ns)) {
          abort_flag = 1;
          atomicOr(p.status, 1);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = su32(sRing + st * stage_bytes);
        const uint32_t b0s = su32(sR + (size_t)kb * NR * 128);
        const uint32_t tmem_d = tmem_acc + (uint32_t)(kb % NACC) * kAccStride;
#pragma unroll
        for (int k = 0; k < SK / 16; ++k)
          tc_mma(tmem_d, desc_sw128(a0 + k * 32), desc_sw128(b0s + k * 32), idesc, (kb >= NACC) || (k != 0));
        tc_commit(su32(&bars[SMAXST + st]));
        if (++st == nstages) {
          st = 0;
          ph ^= 1u;
        }
      }
      tc_commit(su32(&bars[2 * SMAXST]));  // accumulator of step s complete
    }
    // every thread advances the ring position the same way
    for (int kb = 0; kb < KB; ++kb)
      if (++stage == nstages) {
        stage = 0;
        phase ^= 1u;
      }

    // ---- gate warps: wait for the accumulator, then the gate arithmetic
    if (gate_warp) {
      if (!abort_flag && !bar_wait(su32(&bars[2 * SMAXST]), (uint32_t)(s & 1), p.timeout_ns)) {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
      tc_fence_after();
      // sum of the accumulators in a fixed order: ((a0 + a1) + (a2 + a3))
      uint32_t acc[NCOL];
      {
        const uint32_t ta = tmem_acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(uh0 * G);
        const int nacc = KB < NACC ? KB : NACC;
        float sum01[NCOL], sum23[NCOL];
        uint32_t t0[NCOL];
        tmem_ld<NCOL>(ta, t0);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) sum01[i] = __uint_as_float(t0[i]);
        if (nacc > 1) {
          tmem_ld<NCOL>(ta + kAccStride, t0);
#pragma unroll
          for (int i = 0; i < NCOL; ++i) sum01[i] += __uint_as_float(t0[i]);
        }
        if (nacc > 2) {
          tmem_ld<NCOL>(ta + 2 * kAccStride, t0);
#pragma unroll
          for (int i = 0; i < NCOL; ++i) sum23[i] = __uint_as_float(t0[i]);
          if (nacc > 3) {
            tmem_ld<NCOL>(ta + 3 * kAccStride, t0);
#pragma unroll
            for (int i = 0; i < NCOL; ++i) sum23[i] += __uint_as_float(t0[i]);
          }
#pragma unroll
          for (int i = 0; i < NCOL; ++i) sum01[i] += sum23[i];
        }
#pragma unroll
        for (int i = 0; i < NCOL; ++i) acc[i] = __float_as_uint(sum01[i]);
      }
      const bool active = s < len;
      const int t = active ? (reverse ? len - 1 - s : s) : s;
      float hn[UH];
#pragma unroll
      for (int u = 0; u < UH; ++u) {
        const int c = (uh0 + u) * G;
        float pre[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pre[g] = ((xv[u * G + g] + __uint_as_float(acc[u * G + g])) + wb_s[c + g]) + rb_s[c + g];
        hn[u] = hreg[u];
        if constexpr (CELL == 0) {
          // rows u*4 + g: i, o, f, c
          float pi = pre[0], po = pre[1], pf = pre[2], pc = pre[3];
          if (has_p) {
            pi = pi + pp_s[(uh0 + u) * 3 + 0] * creg[u];
            pf = pf + pp_s[(uh0 + u) * 3 + 2] * creg[u];
          }
          const float ig = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pi));
          const float fg = input_forget ? 1.0f - ig : act<GEN, 0>(p, d * A + 0, clip_pre(clip, pf));
          const float cg = act<GEN, 1>(p, d * A + 1, clip_pre(clip, pc));
          const float cn = fg * creg[u] + ig * cg;
          if (has_p) po = po + pp_s[(uh0 + u) * 3 + 1] * cn;
          const float og = act<GEN, 0>(p, d * A + 0, clip_pre(clip, po));
          if (active) {
            hn[u] = og * act<GEN, 1>(p, d * A + 2, cn);
            creg[u] = cn;
          }
        } else if constexpr (CELL == 1) {
          // linear_before_reset = 1: h~ = g((xw_h + r*(rec_h + Rb_h)) + Wb_h)
          const float z = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[0]));
          const float r = act<GEN, 0>(p, d * A + 0, clip_pre(clip, pre[1]));
          const float ph = (xv[u * G + 2] + r * (__uint_as_float(acc[u * G + 2]) + rb_s[c + 2])) + wb_s[c + 2];
          const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ph));
          if (active) hn[u] = (1.0f - z) * hc + z * hreg[u];
        } else {
          if (active) hn[u] = act<GEN, 1>(p, d * A + 0, clip_pre(clip, pre[0]));
        }
      }
      if (grow) {
        // the 8 units are one 16-byte chunk of their k block's row br
        const int jb = j0 + uh0;
        __half* hdst = reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(h16 + h16_block(p, nxt, d, tin, jb / SK, KB, box_rows)) +
                                                 sw128_offset(br, jb % SK));
        __half* ydst = Y != nullptr ? Y + y_index(p, t, d, bg, jb) : nullptr;
        __align__(16) __half hv[UH], yv[UH];
#pragma unroll
        for (int u = 0; u < UH; ++u) {
          const bool in = jb + u < H;
          if (in) hreg[u] = hn[u];
          hv[u] = __float2half_rn(in ? hn[u] : 0.0f);
          yv[u] = __float2half_rn(active ? hn[u] : 0.0f);
        }
        if (s + 1 < Tn) *reinterpret_cast<uint4*>(hdst) = *reinterpret_cast<const uint4*>(hv);
        if (ydst != nullptr) {
          if (jb + UH <= H && (reinterpret_cast<uintptr_t>(ydst) & 15) == 0) {
            *reinterpret_cast<uint4*>(ydst) = *reinterpret_cast<const uint4*>(yv);
          } else {
            for (int u = 0; u < UH; ++u)
              if (jb + u < H) ydst[u] = yv[u];
          }
        }
      }
      load_xw(s + 1, xv);
      tc_fence_before();
    }
    if (s + 1 < Tn) {
      // the new h copies are read next step by TMA (async proxy) in other CTAs
      asm volatile("fence.proxy.async.global;" ::: "memory");
      alive = team_barrier(p.counters + team, (unsigned)C * (++nbar), p.timeout_ns, p.status, &flag_smem) && !abort_flag;
      tc_fence_after();
    }
  }

  // ---------------- outputs: zero Y past the loop, final states
  if (grow && alive && !abort_flag) {
#pragma unroll
    for (int u = 0; u < UH; ++u) {
      const int j = j0 + uh0 + u;
      if (j >= H) continue;
      if (Y != nullptr)
        for (int t = Tn; t < S; ++t) Y[y_index(p, t, d, bg, j)] = __float2half_rn(0.0f);
      const bool zero = S > 0 && len == 0;
      const size_t si = state_index(p, d, bg, j);
      if (p.Yh != nullptr) static_cast<__half*>(p.Yh)[si] = __float2half_rn(zero ? 0.0f : hreg[u]);
      if (CELL == 0 && p.Yc != nullptr) static_cast<__half*>(p.Yc)[si] = __float2half_rn(zero ? 0.0f : creg[u]);
    }
  }
  // drain: copies and MMAs this CTA issued must be complete before it exits
  if (warp == 8 && lane == 0 && abort_flag) {
    for (int i = 0; i < SMAXST; ++i)
      if (armed[i] >= 0) bar_wait(su32(&bars[i]), (uint32_t)armed[i], p.timeout_ns);
  }
  if (warp == 9 && lane == 0) {
    tc_commit(su32(&bars[2 * SMAXST]));
    bar_wait(su32(&bars[2 * SMAXST]), (uint32_t)(Tn & 1), p.timeout_ns);
  }
  (void)ystride;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_acc), "r"(kTmemCols) : "memory");
  }
}

template <int CELL, bool GEN, bool PLAIN>
cudaError_t step_tc_launch(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16) {
  auto kern = step_tc_kernel<CELL, GEN, PLAIN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  if (resident != nullptr) {
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, STHREADS, plan.smem);
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *resident = (e == cudaSuccess) ? (per_sm * sms) / plan.team_ctas : 0;
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
  cfg.blockDim = dim3(STHREADS, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, h16);
}

template <int CELL>
cudaError_t step_tc_cell(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q, __half* h16) {
  const bool plain = !(p.clip > 0.0f) && p.P == nullptr && !p.input_forget;
  if (p.generic_acts)
    return plain ? step_tc_launch<CELL, true, true>(p, plan, s, q, h16) : step_tc_launch<CELL, true, false>(p, plan, s, q, h16);
  return plain ? step_tc_launch<CELL, false, true>(p, plan, s, q, h16) : step_tc_launch<CELL, false, false>(p, plan, s, q, h16);
}

}  // namespace

size_t step_tc_smem(int G, int H) { return tc_smem_layout(G, H).total; }

cudaError_t step_tc_entry(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, void* h16) {
  __half* hp = static_cast<__half*>(h16);
  switch (p.cell) {
    case 0: return step_tc_cell<0>(p, plan, s, resident, hp);
    case 1: return step_tc_cell<1>(p, plan, s, resident, hp);
    default: return step_tc_cell<2>(p, plan, s, resident, hp);
  }
}

}  // namespace rk
