// Per-token absmax int8 activation quantization ("binary-gemm" card,
// sections "API" quantize_activation and "Correctness"); the formula and its
// binary32 steps are in act_quant.cuh.  Rows that are 16-byte aligned with
// K % 8 == 0 take the register-resident kernel (several tokens per CTA, x
// read once); other shapes take one CTA per token.
#include "act_quant.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

template <bool XB>
__device__ __forceinline__ float load(const void* x, int64_t i) {
  if (XB) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(x)[i]);
  return reinterpret_cast<const float*>(x)[i];
}

// One CTA per token (any K, any alignment).
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

// TT threads per token (a multiple of 32 dividing 256), 256 / TT tokens per
// CTA: thread i of a token holds chunks i, i + TT, ... (8 elements each, at
// most CH of them) in registers, so x is read once; the token's maximum
// meets across its warps in shared memory.  Rows 16-byte aligned, K % 8 == 0.
template <bool XB, int CH>
__global__ void __launch_bounds__(256) act_quant_rows_kernel(const void* __restrict__ x, int M, int K, int TT,
                                                             int8_t* __restrict__ q, float* __restrict__ s) {
  __shared__ float red[8];
  const int tok = threadIdx.x / TT, i = threadIdx.x % TT;
  const int m = blockIdx.x * (256 / TT) + tok;
  const int n8 = K / 8;
  const size_t row_bytes = size_t(K) * (XB ? 2 : 4);
  pdl_wait();
  float v[CH][8];
  float a = 0.f;
  if (m < M) {
    const void* xr = reinterpret_cast<const uint8_t*>(x) + size_t(m) * row_bytes;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int k8 = i + c * TT;
      if (k8 < n8) {
        load8<XB>(xr, k8, v[c]);
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[c][j]));
      }
    }
  }
  a = warp_max(a);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float amax = 0.f;
  for (int w = tok * (TT / 32); w < (tok + 1) * (TT / 32); ++w) amax = fmaxf(amax, red[w]);
  float sc, inv;
  absmax_scales(amax, sc, inv);
  if (m < M) {
    if (i == 0) s[m] = sc;
    uint2* qr = reinterpret_cast<uint2*>(q + size_t(m) * K);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int k8 = i + c * TT;
      if (k8 < n8) qr[k8] = quant8(v[c], inv);
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_act_quant(const void* x, bl_dtype xt, int64_t M, int64_t K, int8_t* q, float* sc, cudaStream_t s) {
  const bool pdl = overlap_enabled();
  const bool xb = xt == BL_BF16;
  const int ch = xb ? 8 : 4;  // chunks a thread keeps in registers
  const bool vec = K % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 && ((K * (xb ? 2 : 4)) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(q) & 7) == 0 && K <= 8 * 256 * ch && M <= 0x7fffffff;
  if (vec) {
    int tt = 32;
    while (tt < 256 && (K / 8 + tt - 1) / tt > ch) tt *= 2;
    const unsigned grid = unsigned((M + 256 / tt - 1) / (256 / tt));
    if (xb) return launch(act_quant_rows_kernel<true, 8>, dim3(grid), dim3(256), 0, s, pdl, x, int(M), int(K), tt, q, sc);
    return launch(act_quant_rows_kernel<false, 4>, dim3(grid), dim3(256), 0, s, pdl, x, int(M), int(K), tt, q, sc);
  }
  if (xb) return launch(act_quant_kernel<true>, dim3(unsigned(M)), dim3(256), 0, s, pdl, x, K, q, sc);
  return launch(act_quant_kernel<false>, dim3(unsigned(M)), dim3(256), 0, s, pdl, x, K, q, sc);
}

}  // namespace bl
