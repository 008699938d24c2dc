// rk_proj.cu -- input projection on SIMT cores: Xw[d] = X . W[d]^T for every
// step and direction at once (web page "Recurrent layers", section "How a
// layer runs", step 1: one batched product, batch = directions, W in the
// transposed-B form; the Gemm page states the float32 accumulation).
//
// X is [M, K] (M = seq * batch rows in X's storage order, K = input), W[d] is
// [N, K] (N = gates * hidden), Xw[d] is [M, N] float32.  Elements are read
// as float or Half and widened; every product and sum is float32 with fused
// multiply-add, one chain per output element in increasing k, so the result
// does not depend on scheduling.
//
// Tiling: a 64 x 64 tile of Xw per 256-thread CTA, k in steps of 16 staged
// through shared memory k-major (so each thread reads its 4 rows and 4
// columns as float4), 4 x 4 outputs per thread.  Loads are bounds-checked and
// element-wise, so any M, N, K and any element offset works.
#include <cuda_fp16.h>

#include "rk_internal.h"

namespace rk {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, PADM = 4;

template <typename T>
__device__ __forceinline__ float widen(T v);
template <>
__device__ __forceinline__ float widen<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen<__half>(__half v) { return __half2float(v); }

template <typename T>
__global__ void __launch_bounds__(256) proj_simt_kernel(int M, int N, int K, const T* __restrict__ X,
                                                         const T* __restrict__ W, float* __restrict__ Xw) {
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

}  // namespace

cudaError_t launch_projection_simt(const ProjParams& p, cudaStream_t s) {
  if (p.M <= 0 || p.N <= 0) return cudaSuccess;
  dim3 grid((unsigned)((p.N + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM), (unsigned)p.D);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  if (p.dtype == 0) {
    proj_simt_kernel<float><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const float*>(p.X),
                                                  static_cast<const float*>(p.W), p.Xw);
  } else {
    proj_simt_kernel<__half><<<grid, 256, 0, s>>>(p.M, p.N, p.K, static_cast<const __half*>(p.X),
                                                   static_cast<const __half*>(p.W), p.Xw);
  }
  return cudaGetLastError();
}

}  // namespace rk
