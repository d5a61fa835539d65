// Per-token absmax int8 activation quantization, device pieces shared by the
// stand-alone kernel (act_quant.cu) and the W1A8 kernels that fuse it into
// their prologue ("binary-gemm" card, sections "API" quantize_activation and
// "Correctness").  The card states per-token absmax with under 1%
// reconstruction error; the formula is this library's reading, computed in
// binary32 with round-to-nearest-even:
//   amax = max_k |x[m,k]|;  amax == 0 -> q = 0, s = 0;
//   inv  = 127 / amax;  q = clamp(rint(x * inv), -127, 127);  s = amax / 127.
// Division and multiplication use the _rn intrinsics so that no fused or
// approximate operation changes a rounding; every user calls these helpers,
// so fused and stand-alone quantization give the same bits.
#pragma once
#include "bl_device.cuh"

namespace bl {

__device__ __forceinline__ void absmax_scales(float amax, float& s, float& inv) {
  inv = amax == 0.f ? 0.f : __fdiv_rn(127.0f, amax);
  s = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.0f);
}

__device__ __forceinline__ int quant_code(float v, float inv) {
  float r = rintf(__fmul_rn(v, inv));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return int(r);
}

// Eight consecutive activations of a row at element 8*i, as fp32 (16-byte
// aligned row; bf16 widened exactly).
template <bool XB>
__device__ __forceinline__ void load8(const void* xr, int64_t i, float (&v)[8]) {
  if (XB) {
    const uint4 u = reinterpret_cast<const uint4*>(xr)[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
    const float4 a = reinterpret_cast<const float4*>(xr)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(xr)[2 * i + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// The eight int8 codes of load8's elements, packed little-endian in two words.
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float inv) {
  uint32_t b[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j >> 2] |= (uint32_t(quant_code(v[j], inv)) & 0xffu) << (8 * (j & 3));
  return make_uint2(b[0], b[1]);
}

// Block-wide scales of the MT tokens of x [MT, K] (K % 8 == 0, rows 16-byte
// aligned): every thread of the block calls it; `red` holds 32 * MT floats.
// Ends with a block barrier, after which scale[m] and inv[m] are valid.
template <int MT, bool XB>
__device__ __forceinline__ void token_scales(const void* x, int64_t K, float* red, float* scale, float* inv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  const int64_t n8 = K / 8;
  const size_t row_bytes = size_t(K) * (XB ? 2 : 4);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const void* xr = reinterpret_cast<const uint8_t*>(x) + m * row_bytes;
    float a = 0.f;
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n8; i += blockDim.x) {
      float v[8];
      load8<XB>(xr, i, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[j]));
    }
    a = warp_max(a);
    if (lane == 0) red[warp * MT + m] = a;
  }
  __syncthreads();
  if (threadIdx.x < MT) {
    const int m = threadIdx.x;
    float amax = 0.f;
    for (int w = 0; w < nw; ++w) amax = fmaxf(amax, red[w * MT + m]);
    absmax_scales(amax, scale[m], inv[m]);
  }
  __syncthreads();
}

}  // namespace bl
