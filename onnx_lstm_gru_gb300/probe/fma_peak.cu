// fma_peak.cu -- measurement aid, not part of the layer library: a kernel
// that issues nothing but independent float32 fused multiply-adds, so its
// rate is the SMs' float32 FMA throughput (the roof of the float32 SIMT
// kernels).  Each thread runs 8 independent chains x 16 unrolled rounds per
// iteration; a and b come from the host so nothing folds at compile time, and
// the sum is stored only when it equals a value it never takes, so the work
// cannot be removed.  Built into its own shared object.
#include <cuda_runtime.h>

namespace {

constexpr int kChains = 8, kRounds = 16;

__global__ void __launch_bounds__(256) fma_peak_kernel(float* out, int iters, float a, float b) {
  float x[kChains];
#pragma unroll
  for (int i = 0; i < kChains; ++i) x[i] = (float)threadIdx.x * 1e-3f + (float)i;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < kRounds; ++r)
#pragma unroll
      for (int i = 0; i < kChains; ++i) x[i] = fmaf(x[i], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) s += x[i];
  if (s == -1.2345e30f) out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" {

// FLOPs one launch performs (2 per FMA).
double rk_probe_fma_flops(int blocks, int threads, int iters) {
  return 2.0 * kChains * kRounds * (double)iters * (double)blocks * (double)threads;
}

// Enqueue one launch on `stream`; out needs blocks * threads floats (never
// written in practice).  Returns a cudaError_t.
int rk_probe_fma_launch(float* out, int blocks, int threads, int iters, void* stream) {
  if (blocks <= 0 || threads <= 0 || threads > 256 || threads % 32 != 0 || iters <= 0) return (int)cudaErrorInvalidValue;
  fma_peak_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(out, iters, 0.9999999f, 1e-7f);
  return (int)cudaGetLastError();
}

}  // extern "C"
