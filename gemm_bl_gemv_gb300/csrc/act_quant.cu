// Per-token absmax int8 activation quantization ("binary-gemm" card,
// sections "API" quantize_activation and "Correctness"), one CTA per token;
// the formula and its binary32 steps are in act_quant.cuh.
#include "act_quant.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

template <bool XB>
__device__ __forceinline__ float load(const void* x, int64_t i) {
  if (XB) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(x)[i]);
  return reinterpret_cast<const float*>(x)[i];
}

// One CTA per token.
template <bool XB>
__global__ void __launch_bounds__(256) act_quant_kernel(const void* __restrict__ x, int64_t K, int8_t* __restrict__ q,
                                                        float* __restrict__ s) {
  __shared__ float red[8];
  __shared__ float s_inv;
  const int64_t m = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t base = m * K;
  pdl_wait();
  float a = 0.f;
  for (int64_t k = tid; k < K; k += blockDim.x) a = fmaxf(a, fabsf(load<XB>(x, base + k)));
  a = warp_max(a);
  if ((tid & 31) == 0) red[tid >> 5] = a;
  __syncthreads();
  if (tid == 0) {
    float amax = 0.f;
    for (int w = 0; w < int(blockDim.x / 32); ++w) amax = fmaxf(amax, red[w]);
    float sc, iv;
    absmax_scales(amax, sc, iv);
    s_inv = iv;
    s[m] = sc;
  }
  __syncthreads();
  const float inv = s_inv;
  for (int64_t k = tid; k < K; k += blockDim.x) {
    q[base + k] = int8_t(quant_code(load<XB>(x, base + k), inv));
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_act_quant(const void* x, bl_dtype xt, int64_t M, int64_t K, int8_t* q, float* sc, cudaStream_t s) {
  const bool pdl = overlap_enabled();
  if (xt == BL_BF16) return launch(act_quant_kernel<true>, dim3(unsigned(M)), dim3(256), 0, s, pdl, x, K, q, sc);
  return launch(act_quant_kernel<false>, dim3(unsigned(M)), dim3(256), 0, s, pdl, x, K, q, sc);
}

}  // namespace bl
