// rk_noalloc.cu -- fixed device scratch for rk_encode_noalloc.
//
// Some callers cannot call cudaMalloc: a runtime whose memory planner owns
// every device allocation and forbids new ones once it has started, a host
// process with a fixed device-memory budget, or code that must not pay the
// device-wide synchronisation cudaFree can imply.  For them the layer's
// scratch (the float32 projection Xw and the step kernel's exchange buffers,
// barrier counters and status word) lives in this file-scope array instead,
// which every GPU that loads the library holds until the process exits.
//
// In host code `g_noalloc_scratch` names a host-side stand-in, not a device
// address: handing it to a kernel would fault or, where the GPU can reach
// host memory, silently use the wrong memory.  The device address is taken
// with cudaGetSymbolAddress once per device, with that device current, the
// first time rk_encode_noalloc runs on it.
#include <cuda_runtime.h>

#include <mutex>

#include "rk_internal.h"

// 16 MiB of float32 scratch per GPU, and the status word of the step kernel.
static __device__ __align__(256) float g_noalloc_scratch[rk::kNoAllocScratchFloats];
static __device__ int g_noalloc_status;

namespace rk {

namespace {

struct NoAllocDevice {
  bool ready = false;
  float* scratch = nullptr;
  int* status = nullptr;
};

constexpr int kMaxDevices = 64;
NoAllocDevice g_devices[kMaxDevices];
std::mutex g_mutex;

}  // namespace

cudaError_t noalloc_scratch(float** scratch, int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  NoAllocDevice& d = g_devices[dev];
  if (!d.ready) {
    // set-up for this device (it is the current device): device addresses of
    // the two file-scope arrays
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&q, g_noalloc_status);
    if (e != cudaSuccess) return e;
    d.scratch = static_cast<float*>(p);
    d.status = static_cast<int*>(q);
    d.ready = true;
  }
  *scratch = d.scratch;
  *status = d.status;
  return cudaSuccess;
}

}  // namespace rk
