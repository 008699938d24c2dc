// rk_proj_tc.cuh -- the tcgen05 input projection of 16-bit layers (Half or
// bfloat16) as a device routine (web page "Recurrent layers", section "How a
// layer runs", step 1: Xw[d] = X . W[d]^T, one batched product; Fast mode may
// use matrix hardware for Half).  Products of two 16-bit values are exact in
// float32 and the tensor cores accumulate in float32; the order is fixed by
// the tile shape, so runs are bit-identical.  Used by the standalone
// projection kernel (rk_proj_tc.cu) and by the step kernel that computes the
// projection on the SMs the recurrence leaves idle (rk_step_tc.cuh).
//
// X is [M, K] and W is [D*N, K], both of one 16-bit type and K-contiguous
// (K-major operands); Xw is [D, M, N] float32.  Requirements (else the SIMT kernel
// runs): X and W 16-byte aligned, K a multiple of 8 (TMA strides), M, N, K > 0.
//
// One CTA per SM, 192 threads:
//   warp 0  TMA producer: 128 x 64 tile of X and 256 x 64 tile of W per
//           stage (128-byte swizzle), 4 stages, full / empty mbarriers;
//   warp 1  allocates 512 TMEM columns and one lane issues
//           tcgen05.mma.cta_group::1.kind::f16 (M = 128, N = 256, K = 16),
//           four per stage, into one of two 256-column fp32 accumulators;
//           tcgen05.commit frees each stage and publishes each tile;
//   warps 2-5 epilogue: tcgen05.ld 32 columns at a time from their TMEM lane
//           quarter and store the rows of Xw (masked at the edges), then
//           release the accumulator.
// The epilogue of one tile overlaps the MMAs of the next.  Every mbarrier
// wait is bounded by a deadline on %globaltimer; on expiry the CTA sets the
// status word, stops issuing, waits (bounded) for its copies and MMAs in
// flight, frees its TMEM and returns.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "rk_elem.cuh"
#include "rk_internal.h"

namespace rk {
namespace ptc {

constexpr int TBM = 128, TBN = 256, TBK = 64, TSTAGES = 4;
constexpr int TTHREADS = 192;
constexpr uint32_t kStageBytesA = TBM * TBK * 2;  // 16 KB
constexpr uint32_t kStageBytesB = TBN * TBK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 512;               // two 256-column accumulators
static_assert(2 * TBN <= (int)kTmemCols, "both accumulators fit the TMEM allocation");
constexpr size_t kTcSmem = (size_t)TSTAGES * (kStageBytesA + kStageBytesB) + 1024 /* alignment */ + 256 /* barriers */;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint32_t b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(par)
      : "memory");
  return ok != 0;
}
// bounded wait; false on timeout
__device__ __forceinline__ bool bar_wait(uint32_t b, uint32_t par, long long timeout_ns) {
  if (bar_try(b, par)) return true;
  const unsigned long long t0 = gtime();
  for (unsigned it = 1;; ++it) {
    if (bar_try(b, par)) return true;
    if ((it & 15u) == 0 && (long long)(gtime() - t0) > timeout_ns) return false;
  }
}
__device__ __forceinline__ void bar_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzled
// layout TMA writes (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);     // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}
// Instruction descriptor: kind::f16, A and B F16, D F32, both K-major, M = 128, N = 256.
// kind::f16 instruction descriptor: D float32, A and B K-major, M = 128,
// N = 256; the A/B type fields (Half or bfloat16) are or-ed in per layer
constexpr uint32_t kIdescBase = (1u << 4) | ((uint32_t)(TBN >> 3) << 17) | ((uint32_t)(TBM >> 4) << 24);

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The projection's work for one CTA: tiles pb, pb + np, ... of the
// D * mt * nt tiles, tile_of(tile) giving its (direction, first row, first
// column), signal(d, m0) called by lane 0 of each epilogue warp once its 32
// rows of the tile are stored and fenced.  The tile's rows go to rows
// row_of(d, m0) ... of Xw[d] (m0 for the whole Xw; a ring slot otherwise),
// after wait_free(d, m0) (called by lane 0 of each epilogue warp) has
// returned true; false gives up.  tsm: 1024-byte aligned shared
// memory of kTcSmem - 1024 bytes.  idesc: kIdescBase or-ed with the
// element type's A/B fields.  Warps 0-5 take the roles; further warps of the
// block only pass the block-wide barriers.
template <class TileOf, class Signal, class RowOf, class WaitFree>
__device__ __forceinline__ void proj_tc_body(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K,
                                             int D, float* __restrict__ Xw, int vec_store, int* status,
                                             long long timeout_ns, unsigned char* tsm, int pb, int np,
                                             uint32_t idesc, TileOf tile_of, Signal signal, RowOf row_of,
                                             WaitFree wait_free) {
  unsigned char* sA = tsm;
  unsigned char* sB = tsm + TSTAGES * kStageBytesA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + TSTAGES * kStageBytesB);
  // bars: full[4], empty[4], tfull[2], tempty[2], done[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int mt = (M + TBM - 1) / TBM, nt = (N + TBN - 1) / TBN;
  const int ntiles = mt * nt * D;
  const int KB = (K + TBK - 1) / TBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < TSTAGES; ++i) {
      bar_init(su32(&bars[i]), 1);
      bar_init(su32(&bars[4 + i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(su32(&bars[8 + i]), 1);
      bar_init(su32(&bars[10 + i]), 4);
    }
    bar_init(su32(&bars[12]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto give_up = [&]() {
    if (!abort_flag) {
      abort_flag = 1;
      atomicOr(status, 1);
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[TSTAGES];  // parity of the last phase armed per stage, -1 if never
      for (int i = 0; i < TSTAGES; ++i) armed[i] = -1;
      for (int tile = pb; tile < ntiles && !abort_flag; tile += np) {
        const int3 tc = tile_of(tile);
        const int d = tc.x, m0 = tc.y, n0 = tc.z;
        for (int kb = 0; kb < KB; ++kb) {
          if (!bar_wait(su32(&bars[4 + stage]), phase ^ 1u, timeout_ns)) {
            give_up();
            break;
          }
          bar_expect(su32(&bars[stage]), kStageBytesA + kStageBytesB);
          tma_load_2d(su32(sA + stage * kStageBytesA), tmA, kb * TBK, m0, su32(&bars[stage]));
          tma_load_2d(su32(sB + stage * kStageBytesB), tmB, kb * TBK, d * N + n0, su32(&bars[stage]));
          armed[stage] = (int)phase;
          if (++stage == TSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // on a give-up, wait (bounded) for the copies still in flight before the
      // CTA can exit: the last armed phase of every stage must complete
      if (abort_flag) {
        for (int i = 0; i < TSTAGES; ++i)
          if (armed[i] >= 0) bar_wait(su32(&bars[i]), (uint32_t)armed[i], timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      // shared memory stays below 256 KB, so adding address / 16 to the
      // start-address field never carries out of it
      const uint64_t adesc0 = smem_desc_sw128(su32(sA)), bdesc0 = smem_desc_sw128(su32(sB));
      for (int tile = pb; tile < ntiles && !abort_flag; tile += np) {
        if (!bar_wait(su32(&bars[10 + acc]), acc_phase ^ 1u, timeout_ns)) {
          give_up();
          break;
        }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(acc * TBN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!bar_wait(su32(&bars[stage]), phase, timeout_ns)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors differ only in the start-address field (address / 16):
          // advance 16 elements (32 bytes) along K inside the swizzle atom
          const uint64_t ad = adesc0 + (uint64_t)stage * (kStageBytesA >> 4);
          const uint64_t bd = bdesc0 + (uint64_t)stage * (kStageBytesB >> 4);
          tc_mma(tmem_d, ad, bd, idesc, kb != 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < TBK / 16; ++k) tc_mma(tmem_d, ad + 2 * k, bd + 2 * k, idesc, 1u);
          tc_commit(su32(&bars[4 + stage]));  // stage free once these MMAs complete
          if (++stage == TSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(su32(&bars[8 + acc]));  // accumulator complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all issued MMAs complete before TMEM can be freed
      tc_commit(su32(&bars[12]));
      bar_wait(su32(&bars[12]), 0, timeout_ns);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter (warp % 4)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pb; tile < ntiles && !abort_flag; tile += np) {
      const int3 tc = tile_of(tile);
      const int d = tc.x, m0 = tc.y, n0 = tc.z;
      if (!bar_wait(su32(&bars[8 + acc]), acc_phase, timeout_ns)) {
        give_up();
        break;
      }
      int free_ok = 1;
      if (lane == 0) free_ok = wait_free(d, m0) ? 1 : 0;
      __syncwarp();  // lane 0's acquire is ordered before every lane's stores
      if (!__shfl_sync(0xffffffffu, free_ok, 0)) {
        give_up();
        break;
      }
      tc_fence_after();
      const int m = m0 + row;
      float* orow = Xw + ((size_t)d * M + row_of(d, m0) + row) * N;
#pragma unroll 1
      for (int c0 = 0; c0 < TBN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TBN + c0), r);
        const int n = n0 + c0;
        if (m < M) {
          if (vec_store && n + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(orow + n + j) =
                  make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                              __uint_as_float(r[j + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < N) orow[n + j] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        bar_arrive(su32(&bars[10 + acc]));
        __threadfence();  // the warp's stores, seen through __syncwarp, before the signal
        signal(d, m0);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  }
}


}  // namespace ptc
}  // namespace rk
