// rk_step_tc.cuh -- persistent recurrent-step kernel on the tcgen05 tensor
// cores, for 16-bit layers (Half or bfloat16: the element type E) whose
// batch makes R . h a dense product.
//
// What it computes is the same as rk_step.cuh (web page "Recurrent layers",
// sections "How a layer runs" and "Arithmetic and determinism"): per step and
// gate row pre = ((xw + rec) + Wb) + Rb with rec = R_row . h_prev, then
// peepholes, clip, activation and state update (LSTM, RNN, GRU with
// linear_before_reset = 1).  The state (h, c) stays float32 in registers;
// the product's h operand is the state rounded to E, so R (E, exact)
// times that operand is exact in float32 and summed in float32.
//
// Layout: a team per (direction, group of up to 128 batch rows); a team is
// ceil(H / 16) CTAs, each owning 16 hidden units, all CTAs of the launch
// co-resident (cooperative launch).  A CTA keeps its 16 units' G rows of R in
// shared memory, unit-major (row u*G + g), in the 128-byte swizzled K-major
// layout the tensor cores read.  The 16-bit copy of the exchanged h lives in
// global memory as 16 KB regions already in that layout, one 128-row x 64 k
// tile each: for a team of more than 64 rows a region is one 64-wide k block
// of rows 0..127; for a team of at most 64 rows (PAIR) a region holds two
// consecutive k blocks, rows of the even block at tile rows 32 (b % 4) +
// b / 4 and of the odd block 16 rows further, so no tile row is wasted and
// a small batch spreads over the four TMEM lane quarters (the four SM
// sub-partitions that run the gate arithmetic).
// Per step:
//   1. the producer warp copies each region of h_t into a ring of 16 KB
//      stages with one bulk copy, as soon as the CTAs owning it have
//      published it;
//   2. one lane issues tcgen05.mma kind::f16 with M = 128 (tile rows),
//      N = 16 G (the CTA's gate rows), K = 16 per instruction, into fp32 TMEM
//      accumulators (lane = tile row, column = gate row): one accumulator, or
//      with PAIR one for even and one for odd k blocks, each MMA reading the
//      whole tile so that the lanes of the other block's rows hold unused
//      products; operand descriptors are precomputed so issue keeps up with
//      the tensor core; then commits to an mbarrier;
//   3. eight warps read the accumulators with tcgen05.ld (warp w sees lanes
//      32 (w % 4) .. + 31).  Without PAIR thread (w, l) takes batch row
//      32 (w % 4) + l and 8 units; with PAIR lanes l and l + 16 both hold
//      batch row 4 l + w % 4, one the even and one the odd partial sum,
//      they swap halves with a shuffle and take half the units each.  Each thread
//      does the gate arithmetic with its units' c and h in registers and the
//      next step's xw prefetched, writes its piece of the 16-bit copy of the new
//      h and publishes it (proxy fence, then one release add per CTA to the
//      counter of the region its units belong to), then writes Y.
// The three roles run their own loops, linked by mbarriers; no barrier spans
// the CTA or the team inside the step loop.  The summation order is fixed by
// the shape (tensor-core k blocks of 16 in increasing k, then even + odd), so
// runs are bit-identical.  Every wait is bounded; on expiry the kernel sets
// the status word, drains its copies and MMAs, frees its TMEM and returns.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "rk_proj_tc.cuh"
#include "rk_step_common.cuh"

namespace rk {

namespace {

constexpr int SB = 128;          // batch rows per team (MMA M)
constexpr int SK = 64;           // k per ring stage (one 128-byte swizzle atom)
constexpr int SSTAGE = 16 * 1024; // one ring stage: a 128-row x 64 k tile
constexpr int SMAXST = 8;         // most ring stages
constexpr int SJ = 16;           // hidden units per CTA (teams published through region counters)
constexpr int SJC = 32;          // hidden units per CTA of a cluster team
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
// The same wait with cluster-scope acquire, for arrivals from other CTAs.
__device__ __forceinline__ bool bar_wait_cluster(uint32_t b, uint32_t par, long long timeout_ns) {
  auto try_once = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(par)
        : "memory");
    return ok != 0;
  };
  if (try_once()) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (try_once()) return true;
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
// TMEM columns to allocate for `cols` accumulator columns: a power of two, at least 32.
__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t cols) {
  uint32_t n = 32;
  while (n < cols) n <<= 1;
  return n;
}
// kind::f16, D float32, both K-major, M = 128, N = n; the A/B type fields
// (Half or bfloat16, Elem<E>::kMmaAB) are or-ed in by the caller.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(SB >> 4) << 24);
}
// Byte offset of element (row r, k) of a K-major tile of 64-element rows in
// the 128-byte swizzled layout (16-byte chunks of a row XORed with r % 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  const int chunk = (k >> 3) ^ (r & 7);
  return (uint32_t)(r * 128 + chunk * 16 + (k & 7) * 2);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
// NCOL consecutive accumulator columns of this warp's 32 lanes (NCOL a
// multiple of 4), then wait for the loads.
template <int NCOL>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[NCOL]) {
  static_assert(NCOL % 4 == 0, "columns in groups of 4");
  int c = 0;
#pragma unroll
  for (; c + 16 <= NCOL; c += 16) tmem_ld16(taddr + c, r + c);
  if constexpr (NCOL % 16 >= 8) {
    tmem_ld8(taddr + c, r + c);
    c += 8;
  }
  if constexpr (NCOL % 8 == 4) tmem_ld4(taddr + c, r + c);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// UH 16-bit values to 16 (UH = 8) or 8 (UH = 4) aligned bytes.
template <int UH, typename E>
__device__ __forceinline__ void store_halves(E* dst, const E (&v)[UH]) {
  if constexpr (UH == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(v);
  else *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(v);
}
// The same with the streaming cache hint (st.global.cs): for Y, written once
// and not read in the launch, so that its lines leave L2 first and do not
// push out what the launch still reads there (the Xw ring, the exchanged h).
template <int UH, typename E>
__device__ __forceinline__ void store_halves_streaming(E* dst, const E (&v)[UH]) {
  if constexpr (UH == 8) __stcs(reinterpret_cast<uint4*>(dst), *reinterpret_cast<const uint4*>(v));
  else __stcs(reinterpret_cast<uint2*>(dst), *reinterpret_cast<const uint2*>(v));
}


// Shared memory: [R slice: KB blocks of (16 G rows x 64 k) E][ring: stages x 16 KB][barriers][biases]
struct TcSmem {
  size_t r, ring, bar, bias, total;
};
__host__ __device__ inline TcSmem tc_smem_layout(int G, int H, int stages, int sj) {
  TcSmem L{};
  const int KB = (H + SK - 1) / SK;
  const size_t rbytes = (size_t)KB * sj * G * SK * 2;
  size_t o = 1024;  // room to align the dynamic base up to 1024 bytes
  L.r = o;    o += (rbytes + 1023) & ~(size_t)1023;
  L.ring = o; o += (size_t)stages * SSTAGE;
  L.bar = o;  o += 256;
  L.bias = o; o += (size_t)2 * sj * G * 4 + 3 * sj * 4;
  L.total = o;
  return L;
}

// Region (16 KB, 8192 elements) of the 16-bit h copy: buffer, direction, team, region.
__device__ __forceinline__ size_t h16_region(const StepParams& p, int buf, int d, int team_in_dir, int region, int NREG) {
  return ((((size_t)buf * p.D + d) * p.teams_per_dir + team_in_dir) * NREG + region) * (size_t)(SSTAGE / 2);
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// MODE 0: teams of more than 64 rows, one k block per tile, 16 units per
// CTA, published through region counters; MODE 1: teams of at most 64 rows,
// paired k blocks, 16 units per CTA, region counters; MODE 2: as MODE 1 with
// 32 units per CTA and the team one thread-block cluster, published by
// remote mbarrier arrivals instead.
template <int CELL, bool GEN, bool PLAIN, int MODE, typename E>
__global__ void __launch_bounds__(STHREADS, 1) step_tc_kernel(const StepParams p, E* __restrict__ h16,
                                                             const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB) {
  constexpr bool PAIR = MODE >= 1;
  constexpr bool CLU = MODE == 2;
  constexpr int SJT = CLU ? SJC : SJ;  // hidden units per CTA
  constexpr int G = CellInfo<CELL>::G;
  constexpr int A = CellInfo<CELL>::A;
  constexpr int NR = SJT * G;          // gate rows of this CTA (MMA N): 16 to 128
  constexpr int UH = PAIR ? SJT / 4 : SJT / 2;  // units per gate thread: 4 or 8
  constexpr int NCOL = UH * G;         // accumulator values per gate thread
  constexpr int BPR = PAIR ? 2 : 1;    // k blocks per region
  // odd-block accumulator right after the even one, so that with paired
  // blocks one MMA of N = 2 NR (R's blocks 2r and 2r + 1 are adjacent in
  // shared memory) fills both
  constexpr uint32_t kOddCol = PAIR ? (uint32_t)NR : (uint32_t)SJT * 4;
  constexpr uint32_t kTmemCols = tmem_cols_for(2 * kOddCol);  // a power of two >= 32
  static_assert(NR <= (int)kOddCol && 2 * kOddCol <= kTmemCols && kTmemCols <= 512, "accumulators fit the allocation");
  static_assert(!PAIR || (NR % 8 == 0 && 2 * NR <= 256), "paired product: N = 2 NR, whole 8-row swizzle groups");
  extern __shared__ unsigned char tsm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  // projection of the layer computed by the blocks past the recurrence's
  // (flag-published teams, layout 0): tiles in the order the recurrence
  // consumes them (128 rows = time steps, both directions interleaved), each
  // epilogue warp counting its stored rows into the tile's readiness counter
  const int pj_mt = (p.pj_M + ptc::TBM - 1) / ptc::TBM, pj_nt = (G * p.H + ptc::TBN - 1) / ptc::TBN;
  // Xw through a ring of kXwRingTiles 128-row tiles per direction (it stays
  // in L2) when every row has the same length L: both directions then read
  // the tiles strictly one after another, in the order they are produced.
  // Production index k of tile mi: mi forward, pj_mt - 1 - mi reverse; its
  // rows go to ring slot k % ring.  The tile of production index k - ring
  // must have been read by every warp before tile k overwrites it.
  int ring = 0, ring_len = p.T;
  if (MODE != 2 && p.fused && p.xw_ring > 0) {
    bool uniform = true;
    if (p.lens != nullptr) {
      auto clamp_len = [&](int v) {
        v = v < 0 ? 0 : (v > p.S ? p.S : v);
        return v > p.T ? p.T : v;
      };
      ring_len = clamp_len(p.lens[0]);
      for (int b = 1; b < p.N && uniform; ++b) uniform = clamp_len(p.lens[b]) == ring_len;
    }
    ring = uniform ? p.xw_ring : 0;
  }
  auto prod_index = [&](int dd, int mi) {
    const bool rev = p.direction == 1 || (p.direction == 2 && dd == 1);
    return rev ? pj_mt - 1 - mi : mi;
  };
  // the last step that reads a row of tile mi (-1: none), for length ring_len
  auto last_step = [&](int dd, int mi) {
    const bool rev = p.direction == 1 || (p.direction == 2 && dd == 1);
    const int t_lo = (int)(((long long)mi * ptc::TBM) / p.N);
    const int t_hi = (int)(((long long)(mi + 1) * ptc::TBM - 1) / p.N);
    if (t_lo >= ring_len) return -1;
    return rev ? ring_len - 1 - t_lo : (t_hi < ring_len - 1 ? t_hi : ring_len - 1);
  };
  if constexpr (MODE != 2) {
    if (p.fused && (int)blockIdx.x >= p.step_ctas) {
      auto tile_of = [&](int tile) {
        const int mi = tile / (p.D * pj_nt), rem = tile % (p.D * pj_nt);
        const int dd = rem / pj_nt, n = rem % pj_nt;
        const bool rev = p.direction == 1 || (p.direction == 2 && dd == 1);
        return make_int3(dd, (rev ? pj_mt - 1 - mi : mi) * ptc::TBM, n * ptc::TBN);
      };
      auto signal = [&](int dd, int m0) {
        atomicAdd(p.xw_ready + (size_t)dd * p.xw_groups + (m0 / ptc::TBM) / p.xw_mpg, 1u);
      };
      auto row_of = [&](int dd, int m0) {
        return ring ? (prod_index(dd, m0 / ptc::TBM) % ring) * ptc::TBM : m0;
      };
      // the slot's previous tile must have been read by every warp of the
      // direction: each warp counts one per step whose Xw it has loaded
      auto wait_free = [&](int dd, int m0) -> bool {
        if (!ring) return true;
        const int k = prod_index(dd, m0 / ptc::TBM);
        if (k < ring) return true;
        const int kp = k - ring;
        const bool rev = p.direction == 1 || (p.direction == 2 && dd == 1);
        const int sl = last_step(dd, rev ? pj_mt - 1 - kp : kp);
        if (sl < 0) return true;
        const unsigned target = (unsigned)(sl + 1) * (unsigned)p.xw_consumers;
        const unsigned* cnt = p.xw_done + dd;
        if (ld_acquire_gpu(cnt) >= target) return true;
        const unsigned long long t0 = global_ns();
        for (unsigned it = 1;; ++it) {
          if (ld_acquire_gpu(cnt) >= target) return true;
          if ((it & 15u) == 0 && (long long)(global_ns() - t0) > p.timeout_ns) return false;
        }
      };
      ptc::proj_tc_body(&tmA, &tmB, p.pj_M, G * p.H, p.pj_K, p.D, const_cast<float*>(p.xw), p.pj_vec, p.status,
                        p.timeout_ns, base, (int)blockIdx.x - p.step_ctas, (int)gridDim.x - p.step_ctas,
                        ptc::kIdescBase | Elem<E>::kMmaAB, tile_of, signal, row_of, wait_free);
      return;
    }
  }
  const int NST = p.stages;
  const TcSmem L = tc_smem_layout(G, p.H, NST, SJT);
  unsigned char* sR = base + (L.r - 1024);
  unsigned char* sRing = base + (L.ring - 1024);
  // full[8], empty[8], done, pub, free, drain, cluster publication[2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (L.bar - 1024));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SMAXST + 6);
  float* wb_s = reinterpret_cast<float*>(base + (L.bias - 1024));
  float* rb_s = wb_s + NR;
  float* pp_s = rb_s + NR;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, N = p.N, S = p.S, Tn = p.T;
  const int C = p.team_ctas;
  // teams interleaved over the block index: consecutive blocks tend to share
  // a die, and a team spread evenly over both dies keeps a steadier pace
  // than one split unevenly
  const int nteams = (p.fused ? p.step_ctas : (int)gridDim.x) / C;
  int team, rank;
  if constexpr (CLU) {
    // one team per cluster of C CTAs
    team = blockIdx.x / C;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  } else {
    team = blockIdx.x % nteams;
    rank = blockIdx.x / nteams;
  }
  const int d = team / p.teams_per_dir;
  const int tin = team % p.teams_per_dir;  // team index within its direction
  const int b0 = tin * SB;
  const int nbt = min(SB, N - b0);
  const int j0 = rank * SJT;
  const int KB = (H + SK - 1) / SK;
  const int NREG = (KB + BPR - 1) / BPR;  // regions per step
  const bool reverse = p.direction == 1 || (p.direction == 2 && d == 1);
  const size_t GH = (size_t)G * H;
  const E* R = static_cast<const E*>(p.R);
  const E* Bias = static_cast<const E*>(p.Bias);
  const E* P = static_cast<const E*>(p.P);
  const E* h0 = static_cast<const E*>(p.h0);
  const E* c0 = static_cast<const E*>(p.c0);
  E* Y = static_cast<E*>(p.Y);

  // ---------------- prologue: R slice (unit-major rows, swizzled), biases, barriers, TMEM
  // 8 consecutive k (16 bytes) at a time: H is a multiple of 8, so a chunk
  // is wholly inside or wholly past H, and lands as one 16-byte piece of the
  // swizzled row; element loads when R is not 16-byte aligned
  const bool r_vec = (reinterpret_cast<uintptr_t>(R) & 15) == 0;
  for (int e = tid; e < KB * NR * (SK / 8); e += blockDim.x) {
    const int kb = e / (NR * (SK / 8));
    const int rem = e % (NR * (SK / 8));
    const int r = rem / (SK / 8), kk = (rem % (SK / 8)) * 8;
    const int u = r / G, g = r % G, k = kb * SK + kk;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j0 + u < H && k < H) {
      const E* src = R + ((size_t)d * GH + (size_t)g * H + j0 + u) * H + k;
      if (r_vec) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        __align__(16) E t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = src[i];
        v = *reinterpret_cast<const uint4*>(t8);
      }
    }
    *reinterpret_cast<uint4*>(sR + (size_t)kb * NR * 128 + sw128_offset(r, kk)) = v;
  }
  for (int e = tid; e < NR; e += blockDim.x) {
    const int u = e / G, g = e % G;
    const bool ok = j0 + u < H && Bias != nullptr;
    wb_s[e] = ok ? Elem<E>::to_f(Bias[(size_t)d * 2 * GH + (size_t)g * H + j0 + u]) : 0.0f;
    rb_s[e] = ok ? Elem<E>::to_f(Bias[(size_t)d * 2 * GH + GH + (size_t)g * H + j0 + u]) : 0.0f;
  }
  for (int e = tid; e < 3 * SJT; e += blockDim.x) {
    const int u = e / 3, g = e % 3;
    pp_s[e] = (CELL == 0 && !PLAIN && P != nullptr && j0 + u < H) ? Elem<E>::to_f(P[(size_t)d * 3 * H + (size_t)g * H + j0 + u]) : 0.0f;
  }
  if (tid == 0) {
    for (int i = 0; i < SMAXST; ++i) {
      mbar_init(smem_u32(&bars[i]), 1);
      mbar_init(smem_u32(&bars[SMAXST + i]), 1);
    }
    mbar_init(smem_u32(&bars[2 * SMAXST]), 1);      // accumulators complete (MMA commit)
    mbar_init(smem_u32(&bars[2 * SMAXST + 1]), 8);  // gate warps' h copies written
    mbar_init(smem_u32(&bars[2 * SMAXST + 2]), 8);  // gate warps read the accumulators
    mbar_init(smem_u32(&bars[2 * SMAXST + 3]), 1);  // final MMA drain
    // cluster teams: every CTA's publication of h_s, s even / odd
    mbar_init(smem_u32(&bars[2 * SMAXST + 4]), (unsigned)C);
    mbar_init(smem_u32(&bars[2 * SMAXST + 5]), (unsigned)C);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // R was written by ordinary stores; the tensor cores read it through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // gate threads: warps 0..7 (warp w reads TMEM lanes 32 (w % 4) .. + 31)
  const bool gate_warp = warp < 8;
  const int q = warp & 3;
  const bool odd_lane = PAIR && lane >= 16;
  // batch row within the team; with paired blocks row b sits in TMEM lane
  // quarter b % 4, so a small batch spreads over all four sub-partitions
  const int br = PAIR ? 4 * (lane & 15) + q : 32 * q + lane;
  const int uh0 = (warp >> 2) * (SJT / 2) + (odd_lane ? UH : 0);  // first of this thread's units
  const bool grow = gate_warp && br < nbt;
  const int bg = b0 + br;  // global batch row
  float hreg[UH], creg[UH];
  int len = Tn;
  // address of (this thread's batch row, unit j) in buffer buf of the 16-bit h copy
  auto h16_at = [&](int buf, int j) {
    const int kb = j / SK;
    const int row = PAIR ? 32 * (br & 3) + 16 * (kb & 1) + (br >> 2) : br;
    return reinterpret_cast<E*>(reinterpret_cast<unsigned char*>(h16 + h16_region(p, buf, d, tin, kb / BPR, NREG)) +
                                     sw128_offset(row, j % SK));
  };
  if (grow) {
    if (p.lens != nullptr) {
      len = p.lens[bg];
      len = len < 0 ? 0 : (len > S ? S : len);
      len = len > Tn ? Tn : len;
    }
    __align__(16) E hv[UH];
#pragma unroll
    for (int u = 0; u < UH; ++u) {
      const int j = j0 + uh0 + u;
      const size_t si = state_index(p, d, bg, j < H ? j : 0);
      hreg[u] = (j < H && h0 != nullptr) ? Elem<E>::to_f(h0[si]) : 0.0f;
      creg[u] = (CELL == 0 && j < H && c0 != nullptr) ? Elem<E>::to_f(c0[si]) : 0.0f;
      hv[u] = Elem<E>::from_f(j < H ? hreg[u] : 0.0f);  // units past H: the k padding of the product
    }
    store_halves<UH>(h16_at(0, j0 + uh0), hv);  // h_0 into buffer 0
    // k columns past the last CTA's units (up to the 64-wide block) belong to
    // no CTA: zero them once in both buffers (R is zero there too, but a stale
    // Inf or NaN times zero would not be)
    if (rank == C - 1 && uh0 == 0) {
      for (int k = C * SJT; k < KB * SK; ++k)
        for (int buf = 0; buf < 2; ++buf) *h16_at(buf, k) = Elem<E>::from_f(0.0f);
    }
  } else {
#pragma unroll
    for (int u = 0; u < UH; ++u) hreg[u] = creg[u] = 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // cluster teams: every CTA's barriers are initialised before any remote
  // arrival (all CTAs of a cluster run at once and reach this point)
  if constexpr (CLU) asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const uint32_t tmem_acc = *tmem_slot;

  // Region counters: each CTA adds 1 to the counter of the region its units
  // belong to every time it publishes a 16-bit copy of h (h_0 counts as one),
  // so region r holds h_s once its counter reaches (owners of r) * (s + 1).
  // The copy of a region for step s waits for that; no barrier spans the
  // team.  Reusing the two h buffers is safe without one: a CTA writes
  // h_{s+1} only after its product of step s consumed h_s of every CTA, and
  // each CTA published h_s after its own copies of h_{s-1}, the buffer being
  // overwritten, had landed.  Each counter sits on a 128-byte line of its own
  // (in the state scratch after the header, zeroed before the launch): the
  // team's CTAs poll them all every step, and per-CTA flags that shared two
  // lines were measured to delay their detection (median 2.3 against 1.8 us
  // after the last release on the bidirectional 512 x 64 x 1024 Half layer).
  constexpr int RPB = SK * BPR / SJT;  // CTAs owning one region: 4 or 8 (a multiple of 4)
  unsigned* rctr = p.hglob == nullptr ? nullptr
                                      : reinterpret_cast<unsigned*>(p.hglob) + (size_t)team * kTcRegionLines * 32;
  const uint32_t bar_done = su32(&bars[2 * SMAXST]);      // accumulators of a step complete
  const uint32_t bar_pub = su32(&bars[2 * SMAXST + 1]);   // 8 gate-warp arrivals
  const uint32_t bar_free = su32(&bars[2 * SMAXST + 2]);  // accumulators read (8 gate warps)
  const uint32_t bar_drain = su32(&bars[2 * SMAXST + 3]);
  // gate warps: make this CTA's new h copies visible to the async proxy of
  // other CTAs, then thread 0 releases the flag once all 8 warps are in
  // Cluster teams instead arrive (release, cluster scope) on every CTA's
  // publication barrier for h_s, one barrier per step parity: a CTA's
  // arrivals for h_{s+2} come after it saw every arrival for h_{s+1}, each of
  // which its sender made after its own arrivals for h_s, so no barrier can
  // count an arrival of a later step in an earlier phase.
  const uint32_t bar_pubc = su32(&bars[2 * SMAXST + 4]);
  auto publish = [&](unsigned value, uint32_t pub_parity) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_pub) : "memory");
    if constexpr (CLU) {
      // lane q of warp 0 waits for the 8 gate warps itself, then arrives on
      // CTA q's barrier: the C releases go out in parallel
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
    } else if (tid == 0) {
      if (bar_wait(bar_pub, pub_parity, p.timeout_ns)) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(rctr + (size_t)(rank / RPB) * 32) : "memory");
      } else {
        abort_flag = 1;
        atomicOr(p.status, 1);
      }
    }
  };
  uint32_t pub_parity = 0;
  if (gate_warp) publish(1u, pub_parity++ & 1u);

  // xw of this thread's units for step s: Xw[d][m(t, bg)][g*H + j]
  const size_t xw_tstride = p.layout == 0 ? (size_t)N * GH : GH;
  const float* xw_row = p.xw + xw_index(p, d, 0, grow ? bg : 0, 0, 0);
  // the UH units of a gate are contiguous floats: 16-byte loads when they
  // are aligned and all inside H
  const bool xw_vec = (j0 + uh0 + UH <= H) && (H % 4 == 0) && (reinterpret_cast<uintptr_t>(p.xw) % 16 == 0);
  auto load_xw = [&](int s, float (&x)[UH * G]) {
    bool on = grow && s < len && s < Tn;
    const int tt = reverse ? len - 1 - s : s;
    const float* qx = xw_row + (size_t)tt * xw_tstride;
    if (ring && on) {
      // the row's place in its tile's ring slot (layout 0: row tt * N + bg)
      const int m = tt * N + bg, mi = m / ptc::TBM;
      qx = p.xw + ((size_t)d * p.pj_M + (size_t)(prod_index(d, mi) % ring) * ptc::TBM + (m % ptc::TBM)) * GH;
    }
    if (MODE != 2 && p.fused && on) {
      // the blocks computing the projection must have stored this row's
      // 128-row tile of Xw for every column (layout 0: row tt * N + bg)
      const int mtile = (tt * N + bg) / ptc::TBM;
      const int grp = mtile / p.xw_mpg;
      const unsigned target = (unsigned)(min(p.xw_mpg, pj_mt - grp * p.xw_mpg) * pj_nt * 4);
      const unsigned* cnt = p.xw_ready + (size_t)d * p.xw_groups + grp;
      if (ld_acquire_gpu(cnt) < target) {
        const unsigned long long t0 = global_ns();
        for (unsigned it = 1; ld_acquire_gpu(cnt) < target; ++it) {
          if (abort_flag || ((it & 15u) == 0 && (long long)(global_ns() - t0) > p.timeout_ns)) {
            abort_flag = 1;
            atomicOr(p.status, 1);
            on = false;
            break;
          }
        }
      }
    }
    // Xw written during this launch is read with coherent loads
    auto ld = [&](const float* a) { return (MODE != 2 && p.fused) ? __ldcg(a) : __ldg(a); };
    auto ld4 = [&](const float* a) {
      return (MODE != 2 && p.fused) ? __ldcg(reinterpret_cast<const float4*>(a)) : __ldg(reinterpret_cast<const float4*>(a));
    };
    if (on && xw_vec) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int v = 0; v < UH / 4; ++v) {
          const float4 a = ld4(qx + (size_t)g * H + j0 + uh0 + 4 * v);
          x[(4 * v + 0) * G + g] = a.x;
          x[(4 * v + 1) * G + g] = a.y;
          x[(4 * v + 2) * G + g] = a.z;
          x[(4 * v + 3) * G + g] = a.w;
        }
    } else {
#pragma unroll
      for (int u = 0; u < UH; ++u)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int j = j0 + uh0 + u;
          x[u * G + g] = (on && j < H) ? ld(qx + (size_t)g * H + j) : 0.0f;
        }
    }
  };
  const bool has_p = !PLAIN && CELL == 0 && P != nullptr;
  const float clip = PLAIN ? 0.0f : p.clip;
  const bool input_forget = !PLAIN && p.input_forget;

  // Regions are taken in a fixed order per CTA, starting after the region
  // this CTA helps write, so that one late region does not hold up the
  // product of the others; the order (hence the summation order of each
  // unit) depends only on the CTA's rank.
  const int rot = (rank / RPB + 1) % NREG;

  if (warp == 8) {
    // ---------------- producer warp: lane l polls the counter of region l
    // with acquire loads (as fast as relaxed ones here, while a relaxed poll
    // followed by an acquire fence cost about 0.8 us more per detection),
    // then one bulk copy per ready region, in this CTA's order
    int armed[SMAXST];
    for (int i = 0; i < SMAXST; ++i) armed[i] = -1;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int s = 0; s < Tn && ok; ++s) {
      const unsigned want = (unsigned)s + 1u;
      const unsigned long long t0 = global_ns();
      unsigned taken = 0;  // regions copied this step (bit r)
      int pos = 0;         // regions issued so far, in this CTA's order
      if constexpr (CLU) {
        // every CTA of the cluster has published h_s: all regions are ready
        bool okc = true;
        if (lane == 0) okc = bar_wait_cluster(bar_pubc + 8u * (uint32_t)(s & 1), (uint32_t)((s >> 1) & 1), p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, okc ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      while (pos < NREG && ok) {
        bool rd = true;
        if (!CLU && lane < NREG && !((taken >> lane) & 1u)) {
          const int owners = min(C, (lane + 1) * RPB) - lane * RPB;
          rd = ld_acquire_gpu(rctr + (size_t)lane * 32) >= (unsigned)owners * want;
        }
        const unsigned ready = __ballot_sync(0xffffffffu, rd) | taken;
        int end = pos;
        while (end < NREG) {
          int r = end + rot;
          r = r >= NREG ? r - NREG : r;
          if (!((ready >> r) & 1u)) break;
          ++end;
        }
        __syncwarp();
        if (end == pos) {
          const bool give_up = lane == 0 && (abort_flag || (long long)(global_ns() - t0) > p.timeout_ns);
          if (__any_sync(0xffffffffu, give_up)) ok = false;
          continue;
        }
        if (lane == 0) {
          // the owners' generic-proxy stores, acquired above, are read by the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (; pos < end; ++pos) {
          int r = pos + rot;
          r = r >= NREG ? r - NREG : r;
          taken |= 1u << r;
          if (lane == 0) {
            if (bar_wait(su32(&bars[SMAXST + st]), ph ^ 1u, p.timeout_ns)) {
              bar_expect(su32(&bars[st]), SSTAGE);
              bulk_load(su32(sRing + st * SSTAGE), h16 + h16_region(p, s & 1, d, tin, r, NREG), SSTAGE, su32(&bars[st]));
              armed[st] = (int)ph;
            } else {
              ok = false;
            }
          }
          if (++st == NST) {
            st = 0;
            ph ^= 1u;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (!ok && lane == 0) {
      abort_flag = 1;
      atomicOr(p.status, 1);
    }
    // drain: copies this CTA issued must land before it exits
    if (lane == 0)
      for (int i = 0; i < SMAXST; ++i)
        if (armed[i] >= 0) bar_wait(su32(&bars[i]), (uint32_t)armed[i], p.timeout_ns);
  } else if (warp == 9) {
    // ---------------- MMA lane: acc[128 x NR] += tile[128 x 64] . R_block[NR x 64]^T per k block
    if (lane == 0) {
      // only the start-address field (address / 16, bits 0-13) differs
      // between the MMAs' descriptors; every address stays below 256 KB
      const uint32_t idesc = idesc_f16(NR) | Elem<E>::kMmaAB;
      // paired blocks with an even block count: every region has both
      // blocks, and one N = 2 NR product per 16 k fills the even and the odd
      // accumulator at once (fewer, wider MMAs: the issue cost per MMA
      // hardly grows with N); each accumulator gets the same products in
      // the same order as with two N = NR products
      const bool wide = PAIR && (KB % 2 == 0);
      const uint32_t idesc2 = idesc_f16(2 * NR) | Elem<E>::kMmaAB;
      const uint64_t adesc0 = desc_sw128(su32(sRing));
      const uint64_t bdesc0 = desc_sw128(su32(sR));
      constexpr uint64_t kK16 = 32 >> 4;                      // 16 elements of k
      constexpr uint64_t kStageD = SSTAGE >> 4;
      constexpr uint64_t kBlockD = (uint64_t)NR * 128 >> 4;  // one k block of R
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int s = 0; s < Tn && ok; ++s) {
        // the gate warps must have read the previous step's accumulators
        if (s > 0 && !bar_wait(bar_free, (uint32_t)((s - 1) & 1), p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool odd_started = false;
        for (int pos = 0; pos < NREG; ++pos) {
          int r = pos + rot;
          r = r >= NREG ? r - NREG : r;
          if (abort_flag || !bar_wait(su32(&bars[st]), ph, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)st * kStageD;
          uint64_t bd = bdesc0 + (uint64_t)(r * BPR) * kBlockD;
          // the first MMA of each accumulator in a step overwrites it; with
          // an odd number of k blocks the last region has no odd block, and
          // it may come first in this CTA's order
          if (wide) {
            tc_mma(tmem_acc, ad, bd, idesc2, pos != 0 ? 1u : 0u);
            tc_mma(tmem_acc, ad + kK16, bd + kK16, idesc2, 1u);
            tc_mma(tmem_acc, ad + 2 * kK16, bd + 2 * kK16, idesc2, 1u);
            tc_mma(tmem_acc, ad + 3 * kK16, bd + 3 * kK16, idesc2, 1u);
            tc_commit(su32(&bars[SMAXST + st]));
            if (++st == NST) {
              st = 0;
              ph ^= 1u;
            }
            continue;
          }
          tc_mma(tmem_acc, ad, bd, idesc, pos != 0 ? 1u : 0u);
          tc_mma(tmem_acc, ad + kK16, bd + kK16, idesc, 1u);
          tc_mma(tmem_acc, ad + 2 * kK16, bd + 2 * kK16, idesc, 1u);
          tc_mma(tmem_acc, ad + 3 * kK16, bd + 3 * kK16, idesc, 1u);
          bd += kBlockD;
          if (PAIR && 2 * r + 1 < KB) {
            tc_mma(tmem_acc + kOddCol, ad, bd, idesc, odd_started ? 1u : 0u);
            tc_mma(tmem_acc + kOddCol, ad + kK16, bd + kK16, idesc, 1u);
            tc_mma(tmem_acc + kOddCol, ad + 2 * kK16, bd + 2 * kK16, idesc, 1u);
            tc_mma(tmem_acc + kOddCol, ad + 3 * kK16, bd + 3 * kK16, idesc, 1u);
            bd += kBlockD;
            odd_started = true;
          }
          tc_commit(su32(&bars[SMAXST + st]));
          if (++st == NST) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit(bar_done);  // accumulators of step s complete
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
    float xv[UH * G];
    // with the Xw ring: each warp counts one per step whose Xw it has loaded
    auto xw_loaded = [&]() {
      if (!ring) return;
      __syncwarp();
      if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.xw_done + d) : "memory");
    };
    load_xw(0, xv);
    xw_loaded();
    bool ok = true;
    // columns of this warp-half's units (w / 4) * SJT / 2 ... of its 32 lanes;
    // without PAIR the thread's own units
    const uint32_t ta = tmem_acc + ((uint32_t)(q * 32) << 16) + (uint32_t)((PAIR ? (warp >> 2) * (SJT / 2) : uh0) * G);
    for (int s = 0; s < Tn; ++s) {
      if (abort_flag || !bar_wait(bar_done, (uint32_t)(s & 1), p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float acc[NCOL];
      if constexpr (PAIR) {
        // lane l < 16 holds the even-block sums of batch row br, lane l + 16
        // the odd-block sums of the same row; of the warp-half's 2 UH units
        // the even lane takes the first UH and the odd lane the rest, each
        // sending the partner the other half, 4 units at a time
#pragma unroll
        for (int r = 0; r < UH / 4; ++r) {
          uint32_t ea[4 * G], eb[4 * G], oa[4 * G], ob[4 * G];
          tmem_ld<4 * G>(ta + (uint32_t)(4 * r * G), ea);
          tmem_ld<4 * G>(ta + (uint32_t)((UH + 4 * r) * G), eb);
          tmem_ld<4 * G>(ta + kOddCol + (uint32_t)(4 * r * G), oa);
          tmem_ld<4 * G>(ta + kOddCol + (uint32_t)((UH + 4 * r) * G), ob);
#pragma unroll
          for (int i = 0; i < 4 * G; ++i) {
            const float o_a = KB < 2 ? 0.0f : __uint_as_float(oa[i]);  // no odd block
            const float o_b = KB < 2 ? 0.0f : __uint_as_float(ob[i]);
            const float mine = odd_lane ? o_b : __uint_as_float(ea[i]);
            const float give = odd_lane ? o_a : __uint_as_float(eb[i]);
            const float got = __shfl_xor_sync(0xffffffffu, give, 16);
            acc[4 * r * G + i] = odd_lane ? got + mine : mine + got;  // even + odd
          }
        }
      } else {
        uint32_t a[NCOL];
        tmem_ld<NCOL>(ta, a);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) acc[i] = __uint_as_float(a[i]);
      }
      // the accumulators may be overwritten by the next step's product
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_free) : "memory");
      const bool active = s < len;
      const int t = active ? (reverse ? len - 1 - s : s) : s;
      float hn[UH];
#pragma unroll
      for (int u = 0; u < UH; ++u) {
        const int c = (uh0 + u) * G;
        float pre[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pre[g] = ((xv[u * G + g] + acc[u * G + g]) + wb_s[c + g]) + rb_s[c + g];
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
          const float ph = (xv[u * G + 2] + r * (acc[u * G + 2] + rb_s[c + 2])) + wb_s[c + 2];
          const float hc = act<GEN, 1>(p, d * A + 1, clip_pre(clip, ph));
          if (active) hn[u] = (1.0f - z) * hc + z * hreg[u];
        } else {
          if (active) hn[u] = act<GEN, 1>(p, d * A + 0, clip_pre(clip, pre[0]));
        }
      }
      // the UH units are one 8- or 16-byte piece of their k block's row
      const int jb = j0 + uh0;
      __align__(16) E hv[UH], yv[UH];
#pragma unroll
      for (int u = 0; u < UH; ++u) {
        const bool in = jb + u < H;
        if (in) hreg[u] = hn[u];
        hv[u] = Elem<E>::from_f(in ? hn[u] : 0.0f);
        yv[u] = Elem<E>::from_f(active ? hn[u] : 0.0f);
      }
      if (s + 1 < Tn) {
        if (grow) store_halves<UH>(h16_at((s + 1) & 1, jb), hv);
        publish((unsigned)s + 2u, pub_parity++ & 1u);
      }
      if (grow && Y != nullptr) {
        E* ydst = Y + y_index(p, t, d, bg, jb);
        if (jb + UH <= H && (reinterpret_cast<uintptr_t>(ydst) % (2 * UH)) == 0) {
          store_halves_streaming<UH>(ydst, yv);
        } else {
          for (int u = 0; u < UH; ++u)
            if (jb + u < H) ydst[u] = yv[u];
        }
      }
      load_xw(s + 1, xv);
      xw_loaded();
    }
    if (!ok) {
      abort_flag = 1;
      atomicOr(p.status, 1);
    }
    // ---------------- outputs: zero Y past the loop, final states
    if (grow && ok && !abort_flag) {
#pragma unroll
      for (int u = 0; u < UH; ++u) {
        const int j = j0 + uh0 + u;
        if (j >= H) continue;
        if (Y != nullptr)
          for (int t = Tn; t < S; ++t) Y[y_index(p, t, d, bg, j)] = Elem<E>::from_f(0.0f);
        const bool zero = S > 0 && len == 0;
        const size_t si = state_index(p, d, bg, j);
        if (p.Yh != nullptr) static_cast<E*>(p.Yh)[si] = Elem<E>::from_f(zero ? 0.0f : hreg[u]);
        if (CELL == 0 && p.Yc != nullptr) static_cast<E*>(p.Yc)[si] = Elem<E>::from_f(zero ? 0.0f : creg[u]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_acc), "r"(kTmemCols) : "memory");
  }
  // cluster teams: no CTA leaves while a peer may still arrive on its barriers
  if constexpr (CLU) asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int CELL, bool GEN, bool PLAIN, int MODE, typename E>
cudaError_t step_tc_launch(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, E* h16,
                           const CUtensorMap* ta, const CUtensorMap* tb) {
  auto kern = step_tc_kernel<CELL, GEN, PLAIN, MODE, E>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
  cfg.blockDim = dim3(STHREADS, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (MODE == 2) {
    // a team is one cluster; teams never wait on each other
    if (plan.team_ctas > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.team_ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    // teams of CTAs that wait on each other's counters: all resident at once
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (resident != nullptr) {
    if (MODE == 2) {
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      *resident = (e == cudaSuccess) ? n : 0;
      return e;
    }
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, STHREADS, plan.smem);
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *resident = (e == cudaSuccess) ? (per_sm * sms) / plan.team_ctas : 0;
    return e;
  }
  static const CUtensorMap kNoMap{};  // the projection role does not run
  return cudaLaunchKernelEx(&cfg, kern, p, h16, ta != nullptr ? *ta : kNoMap, tb != nullptr ? *tb : kNoMap);
}

template <int MODE, typename E>
cudaError_t step_tc_mode_dispatch(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* q, E* h16,
                                  const CUtensorMap* ta, const CUtensorMap* tb) {
  const bool plain = !(p.clip > 0.0f) && p.P == nullptr && !p.input_forget;
  const bool gen = p.generic_acts != 0;
  switch (p.cell) {
    case 0:
      if (gen) return plain ? step_tc_launch<0, true, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<0, true, false, MODE, E>(p, plan, s, q, h16, ta, tb);
      return plain ? step_tc_launch<0, false, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<0, false, false, MODE, E>(p, plan, s, q, h16, ta, tb);
    case 1:
      if (gen) return plain ? step_tc_launch<1, true, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<1, true, false, MODE, E>(p, plan, s, q, h16, ta, tb);
      return plain ? step_tc_launch<1, false, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<1, false, false, MODE, E>(p, plan, s, q, h16, ta, tb);
    default:
      if (gen) return plain ? step_tc_launch<2, true, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<2, true, false, MODE, E>(p, plan, s, q, h16, ta, tb);
      return plain ? step_tc_launch<2, false, true, MODE, E>(p, plan, s, q, h16, ta, tb) : step_tc_launch<2, false, false, MODE, E>(p, plan, s, q, h16, ta, tb);
  }
}

}  // namespace

// One translation unit per MODE and element type (they compile in parallel).
cudaError_t step_tc_rows(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16,
                         const CUtensorMap* ta, const CUtensorMap* tb);
cudaError_t step_tc_pairs(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16,
                          const CUtensorMap* ta, const CUtensorMap* tb);
cudaError_t step_tc_cluster(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident, __half* h16);
cudaError_t step_tc_rows(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                         __nv_bfloat16* h16, const CUtensorMap* ta, const CUtensorMap* tb);
cudaError_t step_tc_pairs(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                          __nv_bfloat16* h16, const CUtensorMap* ta, const CUtensorMap* tb);
cudaError_t step_tc_cluster(const StepParams& p, const StepPlan& plan, cudaStream_t s, int* resident,
                            __nv_bfloat16* h16);

}  // namespace rk
