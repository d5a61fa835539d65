// Packing kernels (load time): ternary / binary int8 matrices into the i2_s,
// TQ2_0 and W1 containers.  Layouts are documented in include/bl.h.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

// i2_s code of a ternary value ("Hesper/Layers/BitLinear", "i2_s Packing
// Format"): -1 -> 0b00, 0 -> 0b01, +1 -> 0b10 (sign of w decides).
__device__ __forceinline__ uint32_t i2s_code(int8_t w) { return w > 0 ? 2u : (w < 0 ? 0u : 1u); }

// TQ2_0 code ("Hesper/Quantization/TQ2_0", "TQ2_0 Format"): 0 -> 0b00,
// +1 -> 0b01, -1 -> 0b11.
__device__ __forceinline__ uint32_t tq2_code(int8_t w) { return w > 0 ? 1u : (w < 0 ? 3u : 0u); }

// One thread per output word of 4 bytes: bytes p..p+3 of a 32-byte group.
__global__ void pack_i2s_kernel(const int8_t* __restrict__ w, float scale, int64_t N, int64_t K,
                                uint8_t* __restrict__ out) {
  const int64_t words_per_row = K / 16;
  const int64_t total = N * words_per_row;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = i / words_per_row;
    const int64_t j = i % words_per_row;  // word j: group j/8, bytes 4*(j%8) .. +3
    const int8_t* row = w + n * K + (j / 8) * 128 + (j % 8) * 4;
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t byte = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) byte |= i2s_code(row[32 * t + b]) << (6 - 2 * t);
      word |= byte << (8 * b);
    }
    reinterpret_cast<uint32_t*>(out)[i] = word;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<float*>(out + N * (K / 4)) = scale;
}

// One thread per code byte (4 elements) plus one per block for the scale.
__global__ void pack_tq2_0_kernel(const int8_t* __restrict__ w, const uint16_t* __restrict__ d, int64_t N, int64_t K,
                                  uint8_t* __restrict__ out) {
  const int64_t nb = K / 256;
  const int64_t total = N * nb * 65;  // 64 code bytes + 1 scale slot per block
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t blk = i / 65;  // n * nb + b
    const int j = int(i % 65);
    uint8_t* o = out + blk * 66;
    if (j == 64) {
      const uint16_t s = d[blk];
      o[64] = uint8_t(s & 0xFF);
      o[65] = uint8_t(s >> 8);
    } else {
      const int64_t n = blk / nb, b = blk % nb;
      const int8_t* src = w + n * K + b * 256 + 4 * j;
      uint32_t byte = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) byte |= tq2_code(src[e]) << (2 * e);
      o[j] = uint8_t(byte);
    }
  }
}

// One thread per 32-bit word: element k at bit k%32, bit = (w > 0).
__global__ void pack_w1_kernel(const int8_t* __restrict__ w, int64_t N, int64_t K, int32_t* __restrict__ out) {
  const int64_t total = N * (K / 32);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int8_t* src = w + i * 32;
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 32; ++k) word |= (src[k] > 0 ? 1u : 0u) << k;
    out[i] = int32_t(word);
  }
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  const int64_t cap = int64_t(sm_count()) * 32;
  if (g > cap) g = cap;
  return g < 1 ? 1 : int(g);
}

}  // namespace

cudaError_t launch_pack_i2s(const int8_t* w, float scale, int64_t N, int64_t K, uint8_t* out, cudaStream_t s) {
  pack_i2s_kernel<<<grid_for(N * K / 16, 256), 256, 0, s>>>(w, scale, N, K, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_tq2_0(const int8_t* w, const uint16_t* d, int64_t N, int64_t K, uint8_t* out,
                              cudaStream_t s) {
  pack_tq2_0_kernel<<<grid_for(N * (K / 256) * 65, 256), 256, 0, s>>>(w, d, N, K, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_w1(const int8_t* w, int64_t N, int64_t K, int32_t* out, cudaStream_t s) {
  pack_w1_kernel<<<grid_for(N * K / 32, 256), 256, 0, s>>>(w, N, K, out);
  return cudaGetLastError();
}

}  // namespace bl
