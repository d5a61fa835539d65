// Host-side internals of libbl: launch functions called by the C ABI layer.
#pragma once
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bl.h"

namespace bl {

// Overlap (programmatic dependent launch) setting, see bl_set_overlap().
bool overlap_enabled();

// Test limit of the pipeline waits in ns (bl_set_wait_limit), 0 for the
// default; read at launch time by the kernels that honour it.
unsigned long long wait_limit_ns();

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the library's error word on the current device (the
// BL_DEVERR_* bits read by bl_device_error()); kernels receive it as an
// argument.  nullptr if it cannot be resolved.
unsigned int* dev_error_ptr();

// A 2-D tiled TMA descriptor over uint8 [outer][inner] at `base` (16-byte
// aligned) with rows `row_bytes` apart (a multiple of 16), loading boxes of
// box_outer rows x box_inner bytes (box_inner a multiple of 16, both at most
// 256), optionally with the 128-byte swizzle; elements outside the tensor
// read as zero.  Returns false if the driver rejects it.
bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                       uint32_t box_inner, uint32_t box_outer, bool swizzle128);

// Launch plans (geometry, grid, kernel attributes already set) remembered per
// (device, N, K) so that repeated calls skip the occupancy queries.
template <class P>
class PlanCache {
 public:
  bool get(int dev, int64_t N, int64_t K, P* out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < n_; ++i)
      if (e_[i].dev == dev && e_[i].N == N && e_[i].K == K) {
        *out = e_[i].p;
        return true;
      }
    return false;
  }
  void put(int dev, int64_t N, int64_t K, const P& p) {
    std::lock_guard<std::mutex> lock(mu_);
    const int i = n_ < kSize ? n_++ : (next_++ % kSize);
    e_[i] = Entry{dev, N, K, p};
  }

 private:
  static constexpr int kSize = 64;
  struct Entry {
    int dev;
    int64_t N, K;
    P p;
  };
  Entry e_[kSize];
  int n_ = 0, next_ = 0;
  std::mutex mu_;
};

// Set a kernel's dynamic shared memory cap to `bytes` on device `dev` once.
// The cap belongs to the kernel function (not to a launch), so it is set to
// the largest size any plan may use rather than to one plan's size.
cudaError_t raise_smem_cap_impl(const void* kernel, int dev, int bytes);
template <typename... KArgs>
cudaError_t raise_smem_cap(void (*kernel)(KArgs...), int dev, int bytes) {
  return raise_smem_cap_impl(reinterpret_cast<const void*>(kernel), dev, bytes);
}

// Launch helper: cudaLaunchKernelEx with the PDL attribute when overlap is on.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- launchers (validated arguments only) --------------------------------
cudaError_t launch_pack_i2s(const int8_t* w, float scale, int64_t N, int64_t K, uint8_t* out, cudaStream_t s);
cudaError_t launch_pack_tq2_0(const int8_t* w, const uint16_t* d, int64_t N, int64_t K, uint8_t* out, cudaStream_t s);
cudaError_t launch_pack_w1(const int8_t* w, int64_t N, int64_t K, int32_t* out, cudaStream_t s);
cudaError_t launch_act_quant(const void* x, bl_dtype xt, int64_t M, int64_t K, int8_t* q, float* sc, cudaStream_t s);
// residual (y's dtype, [N]) and rms_w (x's dtype, [K]) may be nullptr
cudaError_t launch_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                            int64_t K, cudaStream_t s, const void* residual = nullptr, const void* rms_w = nullptr,
                            float eps = 0.f);
cudaError_t launch_gemv_i2s_gate_up(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x, bl_dtype xt,
                                    void* h, bl_dtype ht, int64_t N, int64_t K, cudaStream_t s);
// The activation-stationary i2_s GEMV (csrc/gemv_i2s_slot.cu): returns
// cudaErrorNotSupported, having launched nothing, for shapes it has no plan
// for; launch_gemv_i2s / launch_gemv_i2s_gate_up then use the tiled kernel.
cudaError_t launch_gemv_i2s_slot(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                                 int64_t K, cudaStream_t s, const void* residual, const void* rms_w, float eps);
cudaError_t launch_gemv_i2s_gate_up_slot(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x,
                                         bl_dtype xt, void* h, bl_dtype ht, int64_t N, int64_t K, cudaStream_t s);
cudaError_t launch_gemv_tq2_0(const uint8_t* packed, const void* x, bl_dtype xt, float* y, int64_t N, int64_t K,
                              cudaStream_t s);
cudaError_t launch_gemm_w1a8(const int8_t* q, const float* sc, const int32_t* wq, const uint16_t* ws,
                             const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                             int32_t* dots, cudaStream_t s);
bool w1a8_rows_applicable(int64_t M, int64_t K, int G);
// One token with 128-element groups (csrc/gemm_w1a8_m1.cu); x != nullptr
// quantizes x (xt) in the kernel instead of taking q and s.  Returns
// cudaErrorNotSupported, having launched nothing, when it has no plan.
bool w1a8_m1_applicable(int64_t M, int64_t N, int64_t K, int G);
cudaError_t launch_gemm_w1a8_m1(const int8_t* q, const float* s, const void* x, bl_dtype xt, const int32_t* wq,
                                const uint16_t* ws, const uint16_t* bias, int64_t N, int64_t K, uint16_t* y,
                                int32_t* dots, cudaStream_t st);
bool w1a8_tc_applicable(int64_t M, int64_t K, int G);
cudaError_t launch_gemm_w1a8_tc(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws,
                                const uint16_t* bias, int64_t M, int64_t N, int64_t K, int G, uint16_t* y,
                                cudaStream_t st);
cudaError_t launch_gemm_w1a8_rows(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws,
                                  const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                  int32_t* dots, cudaStream_t st);
// W1A8 with the per-token act quantization fused in (M <= 8): the
// lane-per-row kernel where it applies, else the tiled kernel.
cudaError_t launch_gemm_w1a8_act(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws,
                                 const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                 cudaStream_t st);
cudaError_t launch_gemm_w1a8_act_tiled(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws,
                                       const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                       cudaStream_t st);
cudaError_t launch_gemm_tq2_0_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N,
                                   int64_t K, float* y, cudaStream_t st);
cudaError_t launch_gemm_i2s_int8_simt(const int8_t* q, const float* sc, const uint8_t* packed, int64_t M, int64_t N,
                                      int64_t K, float* y, int32_t* acc, cudaStream_t s);
cudaError_t launch_gemm_i2s_int8(const int8_t* q, const float* sc, const uint8_t* packed, int64_t M, int64_t N,
                                 int64_t K, float* y, int32_t* acc, cudaStream_t s);
// The prefill from unquantized activations (act quantization fused in); ws
// as laid out by gemm_i2s_int8_act_workspace (barrier words zero before the
// first use).
size_t gemm_i2s_int8_act_workspace(int64_t M, int64_t K);
cudaError_t launch_gemm_i2s_int8_act(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                     int64_t K, float* y, uint8_t* ws, int fuse, cudaStream_t s);
// The same with the workspace in the library's static device array
// (csrc/prefill_noalloc.cu), whose size gemm_i2s_int8_act_noalloc_limit gives.
size_t gemm_i2s_int8_act_noalloc_limit();
cudaError_t launch_gemm_i2s_int8_act_noalloc(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                             int64_t K, float* y, int fuse, cudaStream_t s);

}  // namespace bl
