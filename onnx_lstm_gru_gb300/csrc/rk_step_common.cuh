// rk_step_common.cuh -- what every recurrent-step kernel of this library
// shares (sm_103a): PTX helpers (mbarriers, bulk copies, cluster shared
// memory, release counters, bounded waits), element access, the ONNX
// activations and the clip of the web page "Recurrent layers" (section
// "Arithmetic and determinism"; formulas from the ONNX operator
// definitions), the layout index functions of its section "Layouts", the
// fixed-order warp reduction, and the gate counts of the three cells.
#pragma once

#include <cstdint>

#include "rk_elem.cuh"
#include "rk_internal.h"

namespace rk {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
      "r"(__float_as_uint(v.w)), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(bar)
               : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until the grids this one depends on (programmatic dependent launch)
// have completed and their writes are visible; returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel on the stream, if launched as a programmatic
// dependent, start being scheduled.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait for an mbarrier phase with a deadline.  Returns false on timeout.
// One contiguous global -> shared copy on the async proxy (16-byte aligned
// addresses, size a multiple of 16), counted on mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && (long long)(global_ns() - t0) > timeout_ns) return false;
  }
}

// One arrival (release, CTA scope) on an mbarrier of this CTA.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Poll a counter that writers raise with release adds, with acquire loads,
// until it reaches `target`; false once timeout_ns has passed first.
__device__ __forceinline__ bool counter_wait_bounded(const unsigned* ctr, unsigned target, long long timeout_ns) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    if ((it & 31u) == 0 && (long long)(global_ns() - t0) > timeout_ns) return false;
  }
}

// ------------------------------------------------------------------ element access
template <typename T>
__device__ __forceinline__ float load_elem(const T* p) { return Elem<T>::to_f(*p); }

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v) { *p = Elem<T>::from_f(v); }

// 4 consecutive R elements from shared memory as floats (16-byte aligned rows).
template <typename T>
__device__ __forceinline__ float4 load4_smem(const T* p) { return load4_16(p); }
template <>
__device__ __forceinline__ float4 load4_smem<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// ------------------------------------------------------------------ activations
// sigmoid(x) = 1 / (1 + e^-x) and tanh(x) = 1 - 2 / (e^(2x) + 1), written from
// these identities over the __expf intrinsic and the __fdividef fast
// division.  In float32 both stay within about 1e-6 of the exact value
// (__expf is within a few ulp for the arguments that matter, and the forms
// saturate to 0 / +-1 where the exponential overflows); the parity tests hold
// them to the oracle.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float tanh_fast(float x) { return 1.0f - __fdividef(2.0f, __expf(2.0f * x) + 1.0f); }

// The eleven ONNX activations (the pages name them; formulas from the ONNX
// operator definitions).  Comparisons are written so that NaN passes through.
__device__ __forceinline__ float act_eval(int kind, float a, float b, float x) {
  // a chain of branches on the kind (the same in every thread), not a switch
  if (kind == 0) return sigmoid_fast(x);
  if (kind == 1) return tanh_fast(x);
  if (kind == 7) {
    const float y = a * x + b;
    return y < 0.0f ? 0.0f : (y > 1.0f ? 1.0f : y);
  }
  if (kind == 6) return a * tanh_fast(b * x);
  if (kind == 9) return x / (1.0f + fabsf(x));
  if (kind == 2) return x > 0.0f ? x : (x <= 0.0f ? 0.0f : x);
  if (kind == 3) return a * x + b;
  if (kind == 4) return x >= 0.0f ? x : (x < 0.0f ? a * x : x);
  if (kind == 5) return x > a ? x : (x <= a ? 0.0f : x);
  if (kind == 8) return x >= 0.0f ? x : (x < 0.0f ? a * expm1f(x) : x);
  if (kind == 10) return x > 20.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
  return __int_as_float(0x7fffffff);
}

// The same activations with at most two branches (taken by the whole launch
// alike) instead of one per kind: sigmoid, tanh and scaled tanh share one
// exponential and one fast reciprocal; relu, affine, leaky relu,
// thresholded relu, hard sigmoid and softsign are a few operations each,
// chosen by selects, and never wait for the exponential; ELU and Softplus go
// to act_eval.  Each kind's value comes from the same operations as in
// act_eval (2 * r with r = __fdividef(1, y) equals __fdividef(2, y): the fast
// division multiplies by an approximate reciprocal, and doubling is exact),
// so the two give the same bits.
__device__ __forceinline__ float act_eval_any(int kind, float a, float b, float x) {
  if (kind == 0 || kind == 1 || kind == 6) {
    const float u = kind == 6 ? b * x : x;
    const float e = __expf(kind == 0 ? -u : 2.0f * u);
    const float r = __fdividef(1.0f, 1.0f + e);  // sigmoid(x), or (1 - tanh(u)) / 2
    const float th = 1.0f - 2.0f * r;
    return kind == 0 ? r : (kind == 6 ? a * th : th);
  }
  if (kind < 2 || kind == 8 || kind > 9) return act_eval(kind, a, b, x);
  const float hs = a * x + b;
  float y = x / (1.0f + fabsf(x));  // softsign (9)
  y = kind == 2 ? (x > 0.0f ? x : (x <= 0.0f ? 0.0f : x)) : y;
  y = kind == 3 ? hs : y;
  y = kind == 4 ? (x >= 0.0f ? x : (x < 0.0f ? a * x : x)) : y;
  y = kind == 5 ? (x > a ? x : (x <= a ? 0.0f : x)) : y;
  y = kind == 7 ? (hs < 0.0f ? 0.0f : (hs > 1.0f ? 1.0f : hs)) : y;
  return y;
}

// Slot `slot` of direction d.  GEN = false compiles in the ONNX defaults.
template <bool GEN, int DEFAULT_KIND>
__device__ __forceinline__ float act(const StepParams& p, int idx, float x) {
  if constexpr (GEN) {
    return act_eval(p.acts[idx].kind, p.acts[idx].alpha, p.acts[idx].beta, x);
  } else {
    return act_eval(DEFAULT_KIND, 0.0f, 0.0f, x);
  }
}

// The same with the slot already read into registers (once per launch, so
// that the step loop does not index the parameter array).
template <bool GEN, int DEFAULT_KIND>
__device__ __forceinline__ float act(const ActSlot& a, float x) {
  if constexpr (GEN) {
    return act_eval_any(a.kind, a.alpha, a.beta, x);
  } else {
    return act_eval(DEFAULT_KIND, 0.0f, 0.0f, x);
  }
}

__device__ __forceinline__ float clip_pre(float c, float x) {
  // selects, not branches; NaN passes (every comparison with it is false)
  const float y = x > c ? c : (x < -c ? -c : x);
  return c > 0.0f ? y : x;
}

// ------------------------------------------------------------------ indexing
__device__ __forceinline__ size_t y_index(const StepParams& p, int t, int d, int b, int j) {
  return p.layout == 0 ? (((size_t)t * p.D + d) * p.N + b) * p.H + j
                       : (((size_t)b * p.S + t) * p.D + d) * p.H + j;
}
__device__ __forceinline__ size_t state_index(const StepParams& p, int d, int b, int j) {
  return p.layout == 0 ? ((size_t)d * p.N + b) * p.H + j : ((size_t)b * p.D + d) * p.H + j;
}
__device__ __forceinline__ size_t xw_index(const StepParams& p, int d, int t, int b, int g, int j) {
  const size_t m = p.layout == 0 ? (size_t)t * p.N + b : (size_t)b * p.S + t;
  return (((size_t)d * p.S * p.N + m) * p.G + g) * p.H + j;
}

// ------------------------------------------------------------------ shuffle tree
// Combine N per-lane partial sums across the 32 lanes of a warp.  At each
// level the lanes whose bit is set keep the upper half of the values and the
// others the lower half, so after the levels lane L holds the full sum of
// value index xreduce_index<N>(L) (duplicated across the lanes that differ
// only in bits below 32/N).  Fixed order: deterministic.
template <int N, int O>
__device__ __forceinline__ void xreduce(float* v, int lane) {
  if constexpr (N > 1) {
    constexpr int H2 = N / 2;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < H2; ++i) {
      const float send = up ? v[i] : v[i + H2];
      const float keep = up ? v[i + H2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
    if constexpr (O > 1) xreduce<H2, O / 2>(v, lane);
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
    if constexpr (O > 1) xreduce<1, O / 2>(v, lane);
  }
}
template <int N>
__device__ __forceinline__ int xreduce_index(int lane) {
  int idx = 0, n = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      n >>= 1;
      if (lane & o) idx += n;
    }
  }
  return idx;
}

// ------------------------------------------------------------------ cells
template <int CELL>
struct CellInfo;
template <>
struct CellInfo<0> {  // LSTM: gates i, o, f, c; activations f, g, h
  static constexpr int G = 4, A = 3;
};
template <>
struct CellInfo<1> {  // GRU: gates z, r, h; activations f, g
  static constexpr int G = 3, A = 2;
};
template <>
struct CellInfo<2> {  // RNN: one gate; activation f
  static constexpr int G = 1, A = 1;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

}  // namespace rk
