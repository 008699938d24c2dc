// rk_proj.cu -- input projection on SIMT cores: Xw[d] = X . W[d]^T for every
// step and direction at once (web page "Recurrent layers", section "How a
// layer runs", step 1: one batched product, batch = directions, W in the
// transposed-B form; the Gemm page states the float32 accumulation).
//
// X is [M, K] (M = seq * batch rows in X's storage order, K = input), W[d] is
// [N, K] (N = gates * hidden), Xw[d] is [M, N] float32.  Elements are read
// as float32, Half or bfloat16 and widened; every product and sum is float32
// with fused multiply-add, one chain per output element in increasing k, so
// the result does not depend on scheduling.
//
// Two kernels.  The pipelined one (below) serves 16-byte aligned operands.
// The fallback serves any M, N, K and any element offset: a 64 x 64 tile of
// Xw per 256-thread CTA, k in steps of 16 staged through shared memory
// k-major (so each thread reads its 4 rows and 4 columns as float4), 4 x 4
// outputs per thread, bounds-checked element-wise loads.
#include "rk_elem.cuh"
#include "rk_internal.h"

namespace rk {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, PADM = 4;

template <typename T>
__device__ __forceinline__ float widen(T v) { return Elem<T>::to_f(v); }

template <typename T>
__global__ void __launch_bounds__(256) proj_simt_kernel(int M, int N, int K, const T* __restrict__ X,
                                                         const T* __restrict__ W, float* __restrict__ Xw) {
  // the step kernel after this one may be launched early (programmatic
  // dependent launch); it waits for this grid before reading Xw
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ __align__(16) float As[BK][BM + PADM];
  __shared__ __align__(16) float Bs[BK][BN + PADM];
  const int d = blockIdx.z;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const T* Wd = W + (size_t)d * N * K;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  // staging: thread loads 4 consecutive k of one row of the A tile and of the B tile
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  for (int k0 = 0; k0 < K; k0 += BK) {
    {
      const int m = m0 + lr;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = k0 + lk + e;
        As[lk + e][lr] = (m < M && k < K) ? widen<T>(X[(size_t)m * K + k]) : 0.0f;
      }
      const int n = n0 + lr;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = k0 + lk + e;
        Bs[lk + e][lr] = (n < N && k < K) ? widen<T>(Wd[(size_t)n * K + k]) : 0.0f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = Xw + (size_t)d * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) out[(size_t)m * N + n] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// Pipelined variant for 16-byte aligned operands (X and W bases 16-byte
// aligned, K * element size a multiple of 16): NST stages of 32-deep k tiles
// are kept in flight with cp.async (16-byte copies, zero-filled past M, N
// and K), so the loads of later tiles overlap the arithmetic of earlier ones.
// Tiles are PBM x 64 (PBM = 8, 16, 24 or 32) of Xw per CTA, in one of two
// thread layouts:
//  - rows (grids of several tiles per SM): 128 threads, thread (tm, tn) owns
//    rows tm + 8 i and columns tn + 16 j, j < 4 (small CTAs, several per SM,
//    4 stages);
//  - columns (grids of at most one tile per SM): 256 threads, warp w owns
//    columns 8 w ... 8 w + 7 and lane l column 8 w + l % 8 and rows
//    l / 8 + 4 i (8 warps per SM, 6 stages).  A warp's 16-byte shared loads
//    then touch 4 rows of X and 8 rows of W, one wavefront each, so shared
//    memory feeds twice the products per wavefront of a one-column-per-thread
//    layout with the same warp count (which was bound by shared-load
//    wavefronts).
// Either way the 16-byte loads of a quarter warp hit distinct banks, and each
// output is one fused-multiply-add chain in increasing k.
constexpr int PBN = 64, PBK = 32;

template <typename T>
struct PipeElem {
  static constexpr int per16 = 16 / (int)sizeof(T);  // elements per 16-byte copy
  static constexpr int ld = PBK + per16;             // padded row length (elements)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ float4 load4_row(const T* p) {
  return load4_16(p);
}
template <>
__device__ __forceinline__ float4 load4_row<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

template <bool COLS>
struct PipeLayout {
  static constexpr int threads = COLS ? 256 : 128;
  static constexpr int row_step = COLS ? 4 : 8;  // rows of a thread are r0 + row_step * i
  static constexpr int cols = COLS ? 1 : 4;      // columns per thread
};

template <typename T, int PBM, bool COLS, int NST>
__global__ void __launch_bounds__(PipeLayout<COLS>::threads) proj_pipe_kernel(int M, int N, int K, const T* __restrict__ X,
                                                                            const T* __restrict__ W, float* __restrict__ Xw) {
  static_assert(PBM % 8 == 0 && PBM >= 8 && PBM <= 32, "tile rows: 8 to 32 in steps of 8");
  static_assert(NST >= 2, "at least two stages");
  // the step kernel after this one may be launched early (programmatic
  // dependent launch); it waits for this grid before reading Xw
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using Lay = PipeLayout<COLS>;
  constexpr int THREADS = Lay::threads, CN = Lay::cols, RS = Lay::row_step;
  constexpr int E = PipeElem<T>::per16, LD = PipeElem<T>::ld;
  constexpr int RM = PBM / RS;  // rows per thread
  extern __shared__ __align__(16) unsigned char psm[];
  T* As = reinterpret_cast<T*>(psm);                    // [NST][PBM][LD]
  T* Bs = As + (size_t)NST * PBM * LD;                  // [NST][PBN][LD]
  const int d = blockIdx.z;
  const int m0 = blockIdx.y * PBM, n0 = blockIdx.x * PBN;
  const int tid = threadIdx.x;
  // first row and column of this thread, and the stride between its columns
  const int tm = COLS ? (tid & 31) >> 3 : tid >> 4;
  const int tn = COLS ? (tid >> 5) * 8 + (tid & 7) : tid & 15;
  constexpr int CS = 16;
  const T* Wd = W + (size_t)d * N * K;
  const int KT = (K + PBK - 1) / PBK;
  constexpr int CPR = PBK / E;                          // 16-byte chunks per tile row
  constexpr int A_CH = PBM * CPR, B_CH = PBN * CPR;

  auto issue = [&](int kt) {
    const int st = kt % NST, k0 = kt * PBK;
    for (int c = tid; c < A_CH + B_CH; c += THREADS) {
      const bool isA = c < A_CH;
      const int cc = isA ? c : c - A_CH;
      const int r = cc / CPR, kc = (cc % CPR) * E;
      const int gr = (isA ? m0 : n0) + r;
      const bool ok = gr < (isA ? M : N) && k0 + kc < K;
      const T* src = isA ? X + (size_t)(ok ? gr : 0) * K + (ok ? k0 + kc : 0) : Wd + (size_t)(ok ? gr : 0) * K + (ok ? k0 + kc : 0);
      T* dst = (isA ? As + ((size_t)st * PBM + r) * LD : Bs + ((size_t)st * PBN + r) * LD) + kc;
      cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(dst)), src, ok ? 16 : 0);
    }
  };

  float acc[RM][CN];
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int j = 0; j < CN; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int s = 0; s < NST - 1; ++s) {
    if (s < KT) issue(s);
    cp_async_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<NST - 2>();
    __syncthreads();
    if (kt + NST - 1 < KT) issue(kt + NST - 1);
    cp_async_commit();
    const int st = kt % NST;
    const T* a = As + (size_t)st * PBM * LD;
    const T* b = Bs + (size_t)st * PBN * LD;
#pragma unroll
    for (int kk = 0; kk < PBK; kk += 4) {
      float4 av[RM], bv[CN];
#pragma unroll
      for (int i = 0; i < RM; ++i) av[i] = load4_row<T>(a + (size_t)(tm + RS * i) * LD + kk);
#pragma unroll
      for (int j = 0; j < CN; ++j) bv[j] = load4_row<T>(b + (size_t)(tn + CS * j) * LD + kk);
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < CN; ++j) {
          float x = acc[i][j];
          x = fmaf(av[i].x, bv[j].x, x);
          x = fmaf(av[i].y, bv[j].y, x);
          x = fmaf(av[i].z, bv[j].z, x);
          x = fmaf(av[i].w, bv[j].w, x);
          acc[i][j] = x;
        }
    }
  }
  cp_async_wait<0>();
  float* out = Xw + (size_t)d * M * N;
#pragma unroll
  for (int i = 0; i < RM; ++i) {
    const int m = m0 + tm + RS * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < CN; ++j) {
      const int n = n0 + tn + CS * j;
      if (n < N) out[(size_t)m * N + n] = acc[i][j];
    }
  }
}

template <typename T, int PBM, bool COLS, int NST>
cudaError_t launch_pipe(const ProjParams& p, cudaStream_t s) {
  const size_t smem = (size_t)NST * (PBM + PBN) * PipeElem<T>::ld * sizeof(T);
  auto kern = proj_pipe_kernel<T, PBM, COLS, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.N + PBN - 1) / PBN), (unsigned)((p.M + PBM - 1) / PBM), (unsigned)p.D);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  kern<<<grid, PipeLayout<COLS>::threads, smem, s>>>(p.M, p.N, p.K, static_cast<const T*>(p.X),
                                                     static_cast<const T*>(p.W), p.Xw);
  return cudaGetLastError();
}

template <typename T, bool COLS, int NST>
cudaError_t launch_pipe_rows(const ProjParams& p, cudaStream_t s, int rows) {
  switch (rows) {
    case 8: return launch_pipe<T, 8, COLS, NST>(p, s);
    case 16: return launch_pipe<T, 16, COLS, NST>(p, s);
    case 24: return launch_pipe<T, 24, COLS, NST>(p, s);
    default: return launch_pipe<T, 32, COLS, NST>(p, s);
  }
}

template <typename T>
cudaError_t launch_pipe_for(const ProjParams& p, cudaStream_t s, int rows, bool one_wave) {
  return one_wave ? launch_pipe_rows<T, true, 6>(p, s, rows) : launch_pipe_rows<T, false, 4>(p, s, rows);
}

// ---------------------------------------------------------------------------
// Small grids (web page "Matrix multiplication (Gemm)", section "Small grids
// and few rows").  A product whose tiles cannot fill the GPU leaves most SMs
// idle while each busy one walks a long k; both variants below fix the order
// in which an element's terms are added, so results stay bit-identical from
// run to run.
//
// Split k: each CTA owns a TM x 32 tile of Xw and its 8 warps split k into 4
// ranges (a multiple of 32 terms, at least 64 each) x 2 column halves.  Warp
// (r, c) copies its range of the tile's X rows (shared with the other half)
// and W columns into shared memory with cp.async, chains every one of its
// TM / 8 x 4 outputs over its range in increasing k, and stores the range
// sums; then each output is the sum of its 4 range sums in range order.  The
// ranges replace the page's scratch planes and second pass by shared memory
// inside the CTA, so the whole product is still one launch.
constexpr int SPLIT_RANGES = 4, SPLIT_TN = 32, SPLIT_THREADS = 2 * SPLIT_RANGES * 32;

template <typename T>
struct SplitLayout {
  static constexpr int pad = 16 / (int)sizeof(T);  // 16 bytes between rows: X rows of a quarter warp hit distinct banks
};

// Dynamic shared memory of the split-k kernel.
template <typename T>
size_t split_smem(int TM, int K) {
  const size_t ld = (size_t)K + SplitLayout<T>::pad;
  return ((size_t)TM + SPLIT_TN) * ld * sizeof(T) + (size_t)SPLIT_RANGES * TM * SPLIT_TN * sizeof(float);
}

template <typename T, int TM>
__global__ void __launch_bounds__(SPLIT_THREADS) proj_split_kernel(int M, int N, int K, const T* __restrict__ X,
                                                                   const T* __restrict__ W, float* __restrict__ Xw) {
  static_assert(TM % 8 == 0 && TM >= 8 && TM <= 40, "tile rows: 8 to 40 in steps of 8");
  // the step kernel after this one may be launched early (programmatic
  // dependent launch); it waits for this grid before reading Xw
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) unsigned char ssm[];
  constexpr int E = 16 / (int)sizeof(T);  // elements per 16-byte copy
  constexpr int RI = TM / 8;              // rows per lane
  const int LD = K + SplitLayout<T>::pad;
  T* Xs = reinterpret_cast<T*>(ssm);                    // [TM][LD]
  T* Ws = Xs + (size_t)TM * LD;                         // [32][LD]
  float* Ps = reinterpret_cast<float*>(Ws + (size_t)SPLIT_TN * LD);  // [ranges][TM][32]
  const int d = blockIdx.z;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * SPLIT_TN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = warp >> 1, ch = warp & 1;  // k range, column half
  // range r: [k0, k1), ranges a multiple of 32 terms (the last may be shorter)
  const int KR = ((K + SPLIT_RANGES - 1) / SPLIT_RANGES + 31) & ~31;
  const int k0 = min(K, r * KR), k1 = min(K, k0 + KR);
  const T* Wd = W + (size_t)d * N * K;
  // copies: X rows of this column half's parity, W columns of this half
  const int nch = (k1 - k0) / E;  // K is a multiple of E
  for (int c = lane; c < (TM / 2 + 16) * nch; c += 32) {
    const int row = c / nch, kk = k0 + (c % nch) * E;
    const bool isX = row < TM / 2;
    const int rr = isX ? 2 * row + ch : ch * 16 + (row - TM / 2);
    const int g = (isX ? m0 : n0) + rr;
    const bool ok = g < (isX ? M : N);
    const T* src = (isX ? X : Wd) + (size_t)(ok ? g : 0) * K + kk;
    T* dst = (isX ? Xs : Ws) + (size_t)rr * LD + kk;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // the two warps of range r read each other's X rows
  asm volatile("bar.sync %0, 64;" ::"r"(1 + r) : "memory");
  const int rr0 = lane >> 2, cc = lane & 3;
  float acc[RI][4];
#pragma unroll
  for (int i = 0; i < RI; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k = k0; k < k1; k += 4) {
    float4 xv[RI], wv[4];
#pragma unroll
    for (int i = 0; i < RI; ++i) xv[i] = load4_row<T>(Xs + (size_t)(rr0 + 8 * i) * LD + k);
#pragma unroll
    for (int j = 0; j < 4; ++j) wv[j] = load4_row<T>(Ws + (size_t)(ch * 16 + cc + 4 * j) * LD + k);
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a = acc[i][j];
        a = fmaf(xv[i].x, wv[j].x, a);
        a = fmaf(xv[i].y, wv[j].y, a);
        a = fmaf(xv[i].z, wv[j].z, a);
        a = fmaf(xv[i].w, wv[j].w, a);
        acc[i][j] = a;
      }
  }
#pragma unroll
  for (int i = 0; i < RI; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Ps[((size_t)r * TM + rr0 + 8 * i) * SPLIT_TN + ch * 16 + cc + 4 * j] = acc[i][j];
  __syncthreads();
  float* out = Xw + (size_t)d * M * N;
  for (int e = tid; e < TM * SPLIT_TN; e += SPLIT_THREADS) {
    const int row = e / SPLIT_TN, col = e % SPLIT_TN;
    const int m = m0 + row, n = n0 + col;
    if (m >= M || n >= N) continue;
    float v = Ps[(size_t)row * SPLIT_TN + col];
#pragma unroll
    for (int q = 1; q < SPLIT_RANGES; ++q) v += Ps[((size_t)q * TM + row) * SPLIT_TN + col];
    out[(size_t)m * N + n] = v;
  }
}

template <typename T, int TM>
cudaError_t launch_split_tm(const ProjParams& p, cudaStream_t s) {
  const size_t smem = split_smem<T>(TM, p.K);
  auto kern = proj_split_kernel<T, TM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.N + SPLIT_TN - 1) / SPLIT_TN), (unsigned)((p.M + TM - 1) / TM), (unsigned)p.D);
  kern<<<grid, SPLIT_THREADS, smem, s>>>(p.M, p.N, p.K, static_cast<const T*>(p.X), static_cast<const T*>(p.W), p.Xw);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_split(const ProjParams& p, cudaStream_t s, int tm) {
  switch (tm) {
    case 8: return launch_split_tm<T, 8>(p, s);
    case 16: return launch_split_tm<T, 16>(p, s);
    case 24: return launch_split_tm<T, 24>(p, s);
    case 32: return launch_split_tm<T, 32>(p, s);
    default: return launch_split_tm<T, 40>(p, s);
  }
}

// Tile height of the split-k kernel: the smallest (8 to 40 rows) whose tiles
// fit one wave of one CTA per SM and whose operands fit shared memory; 0 when
// none does (or k is too short to cut into 4 ranges of at least 64 terms).
int split_rows_for(const ProjParams& p, int sms, int eb) {
  if (p.K < SPLIT_RANGES * 64) return 0;
  const long long col_tiles = (long long)((p.N + SPLIT_TN - 1) / SPLIT_TN) * p.D;
  for (int tm = 8; tm <= 40; tm += 8) {
    const long long tiles = col_tiles * ((p.M + tm - 1) / tm);
    const size_t smem = eb == 4 ? split_smem<float>(tm, p.K) : split_smem<__half>(tm, p.K);
    if (tiles <= sms && smem <= 200 * 1024) return tm;
  }
  return 0;
}

// Few rows: at most four rows of X (a layer of one or a few steps of a small
// batch, e.g. decoding one step at a time).  W is stored N x K, so, as the
// page does for that storage, a CTA owns 8 columns, one warp per column, and
// the 32 lanes read consecutive k (lane l takes k = 128 i + 4 l ... + 3, four
// consecutive terms per 8- or 16-byte load): W is streamed once.  Every lane
// chains its terms in increasing k, and one lane per row adds the 32 lane
// sums in lane order through shared memory.
template <typename T, int MR>
__global__ void __launch_bounds__(256) proj_rows_kernel(int M, int N, int K, const T* __restrict__ X,
                                                        const T* __restrict__ W, float* __restrict__ Xw) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float sums[8][MR][32];
  const int d = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  float acc[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
  if (n < N) {
    const T* wrow = W + ((size_t)d * N + n) * K;
    for (int k = 4 * lane; k < K; k += 128) {
      const float4 w = load4_row<T>(wrow + k);
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        if (m >= M) break;
        const float4 x = load4_row<T>(X + (size_t)m * K + k);
        float a = acc[m];
        a = fmaf(x.x, w.x, a);
        a = fmaf(x.y, w.y, a);
        a = fmaf(x.z, w.z, a);
        a = fmaf(x.w, w.w, a);
        acc[m] = a;
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MR; ++m) sums[warp][m][lane] = acc[m];
  __syncwarp();
  if (n < N && lane < M) {
    float v = sums[warp][lane][0];
    for (int l = 1; l < 32; ++l) v += sums[warp][lane][l];
    Xw[((size_t)d * M + lane) * N + n] = v;
  }
}

template <typename T>
cudaError_t launch_rows(const ProjParams& p, cudaStream_t s) {
  dim3 grid((unsigned)((p.N + 7) / 8), (unsigned)p.D, 1);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  proj_rows_kernel<T, 4><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const T*>(p.X), static_cast<const T*>(p.W),
                                               p.Xw);
  return cudaGetLastError();
}

// Tile height: the SM that gets the most tiles sets the time, so take the
// height (8 to 32 rows) that minimises rows x tiles-per-SM, counting 4 rows'
// worth of fixed cost per tile (the loads of W, the prologue).  A grid just
// above the SM count (160 tiles of 16 rows on 152 SMs for the 80 x 1024 x
// 256 bidirectional layer) leaves most SMs idle for the second half.
int pipe_rows_for(long long M, long long col_tiles, int sms) {
  int best = 32;
  long long best_cost = -1;
  for (int rows = 32; rows >= 8; rows -= 8) {
    const long long tiles = col_tiles * ((M + rows - 1) / rows);
    const long long cost = (long long)(rows + 4) * ((tiles + sms - 1) / sms);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = rows;
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_projection_simt(const ProjParams& p, cudaStream_t s) {
  if (p.M <= 0 || p.N <= 0) return cudaSuccess;
  const int eb = p.dtype == 0 ? 4 : 2;
  const bool aligned = (reinterpret_cast<uintptr_t>(p.X) % 16 == 0) && (reinterpret_cast<uintptr_t>(p.W) % 16 == 0) &&
                       ((size_t)p.K * eb) % 16 == 0 && p.K > 0;
  // few rows: 4-element loads need 4-element alignment of both bases and of K
  const bool aligned4 = (reinterpret_cast<uintptr_t>(p.X) % (4 * eb) == 0) &&
                        (reinterpret_cast<uintptr_t>(p.W) % (4 * eb) == 0) && p.K % 4 == 0 && p.K > 0;
  if (p.M <= 4 && aligned4) {
    if (p.dtype == 0) return launch_rows<float>(p, s);
    if (p.dtype == 2) return launch_rows<__nv_bfloat16>(p, s);
    return launch_rows<__half>(p, s);
  }
  if (aligned) {
    int dev = 0, sms = p.sms;
    if (sms <= 0) {
      sms = 148;
      if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int tm = split_rows_for(p, sms, eb);
    if (tm > 0) {
      if (p.dtype == 0) return launch_split<float>(p, s, tm);
      if (p.dtype == 2) return launch_split<__nv_bfloat16>(p, s, tm);
      return launch_split<__half>(p, s, tm);
    }
    const long long col_tiles = (long long)((p.N + PBN - 1) / PBN) * p.D;
    const int rows = pipe_rows_for(p.M, col_tiles, sms);
    const bool one_wave = col_tiles * ((p.M + rows - 1) / rows) <= sms;
    if (p.dtype == 0) return launch_pipe_for<float>(p, s, rows, one_wave);
    if (p.dtype == 2) return launch_pipe_for<__nv_bfloat16>(p, s, rows, one_wave);
    return launch_pipe_for<__half>(p, s, rows, one_wave);
  }
  dim3 grid((unsigned)((p.N + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM), (unsigned)p.D);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  if (p.dtype == 0) {
    proj_simt_kernel<float><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const float*>(p.X),
                                                  static_cast<const float*>(p.W), p.Xw);
  } else if (p.dtype == 2) {
    proj_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const __nv_bfloat16*>(p.X),
                                                          static_cast<const __nv_bfloat16*>(p.W), p.Xw);
  } else {
    proj_simt_kernel<__half><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const __half*>(p.X),
                                                   static_cast<const __half*>(p.W), p.Xw);
  }
  return cudaGetLastError();
}

}  // namespace rk
