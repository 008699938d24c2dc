// rk_proj_tc.cu -- the standalone tcgen05 input projection of 16-bit layers
// (the device routine and its contract are in rk_proj_tc.cuh): a persistent
// kernel over all tiles, and the host side that encodes the tensor maps.
#include "rk_proj_tc.cuh"

namespace rk {

namespace {

using namespace ptc;

__global__ void __launch_bounds__(TTHREADS, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N,
                   int K, int D, float* __restrict__ Xw, int vec_store, int* status, long long timeout_ns,
                   uint32_t idesc) {
  // the step kernel after this one may be launched early (programmatic
  // dependent launch); it waits for this grid before reading Xw
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned char tsm_raw[];
  // 1024-byte aligned stage buffers (128-byte swizzle atoms)
  unsigned char* tsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~(uintptr_t)1023);
  const int mt = (M + TBM - 1) / TBM, nt = (N + TBN - 1) / TBN;
  auto tile_of = [&](int tile) {
    const int d = tile / (mt * nt), rem = tile % (mt * nt);
    return make_int3(d, (rem / nt) * TBM, (rem % nt) * TBN);
  };
  auto no_signal = [](int, int) {};
  auto whole = [](int, int m0) { return m0; };
  auto always_free = [](int, int) { return true; };
  proj_tc_body(&tmA, &tmB, M, N, K, D, Xw, vec_store, status, timeout_ns, tsm, (int)blockIdx.x, (int)gridDim.x,
               idesc, tile_of, no_signal, whole, always_free);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, int dtype) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType ty = dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(map, ty, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool projection_tc_maps(const ProjParams& p, CUtensorMap* a, CUtensorMap* b) {
  return make_map(a, p.X, (uint64_t)p.M, (uint64_t)p.K, TBM, p.dtype) &&
         make_map(b, p.W, (uint64_t)p.D * p.N, (uint64_t)p.K, TBN, p.dtype);
}

size_t projection_tc_smem() { return kTcSmem; }

bool projection_tc_supported(const ProjParams& p) {
  return (p.dtype == 1 || p.dtype == 2) && p.M > 0 && p.N > 0 && p.K > 0 && p.K % 8 == 0 &&
         reinterpret_cast<uintptr_t>(p.X) % 16 == 0 && reinterpret_cast<uintptr_t>(p.W) % 16 == 0;
}

cudaError_t launch_projection_tc(const ProjParams& p, int* status, long long timeout_ns, cudaStream_t s) {
  if (!projection_tc_supported(p)) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!projection_tc_maps(p, &ta, &tb)) return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)((p.M + TBM - 1) / TBM) * ((p.N + TBN - 1) / TBN) * p.D;
  const int grid = (int)(tiles < sms ? tiles : sms);
  const int vec = (reinterpret_cast<uintptr_t>(p.Xw) % 16 == 0) && (p.N % 4 == 0);
  const uint32_t idesc = kIdescBase | (p.dtype == 2 ? Elem<__nv_bfloat16>::kMmaAB : Elem<__half>::kMmaAB);
  proj_tc_kernel<<<grid, TTHREADS, kTcSmem, s>>>(ta, tb, p.M, p.N, p.K, p.D, p.Xw, vec, status, timeout_ns, idesc);
  return cudaGetLastError();
}

}  // namespace rk
