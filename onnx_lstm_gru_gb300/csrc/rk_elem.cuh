// rk_elem.cuh -- the element types a layer's tensors may have: float32,
// IEEE binary16 (Half) and bfloat16.  Every kernel reads elements in their
// storage type, widens them exactly to float32 and computes in float32; an
// output is rounded to its storage type to nearest, ties to even, once.
//
// The recurrent-layers page offers float32 and Half tensors.  bfloat16 comes
// from the web page "Matrix multiplication (Gemm)": its first paragraph lets
// the float32-accumulating product take bfloat16 inputs, and its section
// "Accuracy" bounds that variant at 8e-3 of the largest magnitude (Half:
// 2e-3).  Widening either 16-bit type to float32 is exact, and so is the
// product of two of them in float32, so the tensor-core contractions see the
// stored values unchanged.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace rk {

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};

template <>
struct Elem<__half> {
  // the A and B type fields (bits 7-9 and 10-12) of a kind::f16
  // tcgen05.mma instruction descriptor: 0 selects binary16
  static constexpr uint32_t kMmaAB = 0u;
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
  // two packed elements (low half first) to floats
  static __device__ __forceinline__ float2 pair_to_f(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
  static __device__ __forceinline__ uint32_t pair_from_f(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

template <>
struct Elem<__nv_bfloat16> {
  // A and B type fields of a kind::f16 instruction descriptor: 1 selects bfloat16
  static constexpr uint32_t kMmaAB = (1u << 7) | (1u << 10);
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
  static __device__ __forceinline__ float2 pair_to_f(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  }
  static __device__ __forceinline__ uint32_t pair_from_f(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// 4 consecutive 16-bit elements (8 bytes, 8-byte aligned) as floats.
template <typename T>
__device__ __forceinline__ float4 load4_16(const T* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = Elem<T>::pair_to_f(u.x);
  const float2 b = Elem<T>::pair_to_f(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

}  // namespace rk
