// The i2_s prefill from unquantized activations without a caller workspace:
// bl_gemm_i2s_int8_act with its workspace in this file's static device
// array, for callers that cannot allocate device memory themselves -- code
// that is handed only its input and output pointers by a host program that
// owns all device memory (a plugin, an inference server's callback), or a
// loop that must not call cudaMalloc (it can synchronize the device and can
// fail under memory pressure, neither of which a decode or prefill loop can
// afford).  Nothing here allocates: the array is part of the loaded library
// (every GPU that loads it holds kNoAllocWorkspace bytes until the process
// exits), and its device address is looked up once per device.
#include <cstring>
#include <mutex>

#include "bl_internal.h"

namespace bl {
namespace {

constexpr size_t kNoAllocWorkspace = BL_GEMM_I2S_INT8_ACT_NOALLOC_WORKSPACE;

// The workspace (layout as bl_gemm_i2s_int8_act's): barrier words at byte 0,
// codes at 256, scales after them.  Host code must not use this name as an
// address: it only stands for the device array.
static __device__ __align__(256) uint8_t g_noalloc_ws[kNoAllocWorkspace];

// Device address of g_noalloc_ws on the current device, looked up on the
// first call for that device (with it current); nullptr if the lookup fails.
uint8_t* noalloc_workspace(cudaError_t* err) {
  static uint8_t* cache[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint8_t*>(p);
  }
  return cache[dev];
}

}  // namespace

size_t gemm_i2s_int8_act_noalloc_limit() { return kNoAllocWorkspace; }

cudaError_t launch_gemm_i2s_int8_act_noalloc(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                             int64_t K, float* y, int fuse, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  uint8_t* ws = noalloc_workspace(&e);
  if (!ws) return e;
  // The array keeps the last call's contents.  The codes and scales are
  // rewritten by every call; the grid-barrier count of the single-launch
  // form must start at zero, so it is cleared on the stream first (a call
  // that gave up at the barrier may have left it set).
  if (fuse) {
    e = cudaMemsetAsync(ws, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
  }
  return launch_gemm_i2s_int8_act(x, xt, packed, M, N, K, y, ws, fuse, s);
}

}  // namespace bl
