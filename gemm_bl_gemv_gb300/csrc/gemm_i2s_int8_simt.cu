// i2_s x int8 product on the CUDA cores (exact int32 accumulation with dp4a).
//   acc[m,n] = sum_k q[m,k] w[n,k];   y[m,n] = f32(acc) * s[m] * scale
// ("Hesper/Layers/BitLinear", "BitLinear Mathematics", with int8 activations
// as produced by the per-token absmax quantizer).  Used for small batches
// (M < 64), where a 128-row tensor-core tile would be mostly padding.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kBM = 64, kBN = 64, kBK = 128, kPad = 4;

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__global__ void __launch_bounds__(256) gemm_i2s_int8_simt_kernel(const int8_t* __restrict__ q,
                                                                 const float* __restrict__ s,
                                                                 const uint8_t* __restrict__ packed, int M, int N,
                                                                 int K, float* __restrict__ y,
                                                                 int32_t* __restrict__ acc_out) {
  __shared__ __align__(16) int8_t qs[kBM][kBK + kPad];
  __shared__ __align__(16) int8_t wsm[kBN][kBK + kPad];
  const int tid = threadIdx.x;
  const int tm = tid / 16, tn = tid % 16;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  int acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0;
  pdl_wait();
  for (int k0 = 0; k0 < K; k0 += kBK) {
    // activations: 64 rows x 128 bytes, 32 bytes per thread
    {
      const int r = tid / 4, part = tid % 4;
      uint32_t v[8];
      if (m0 + r < M) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(m0 + r) * K + k0 + 32 * part);
        const uint4 a = src[0], b = src[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) *reinterpret_cast<uint32_t*>(&qs[r][32 * part + 4 * i]) = v[i];
    }
    // weights: one 32-byte i2_s group per row, 8 bytes per thread
    {
      const int r = tid / 4, part = tid % 4;
      uint8_t b[8];
      if (n0 + r < N) {
        const uint2 v = *reinterpret_cast<const uint2*>(packed + int64_t(n0 + r) * (K / 4) + (k0 / 128) * 32 + 8 * part);
#pragma unroll
        for (int i = 0; i < 4; ++i) { b[i] = uint8_t(v.x >> (8 * i)); b[4 + i] = uint8_t(v.y >> (8 * i)); }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = 0x55;  // code 01 = 0
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int p = 8 * part + i;
#pragma unroll
        for (int t = 0; t < 4; ++t) wsm[r][32 * t + p] = int8_t(int((b[i] >> (6 - 2 * t)) & 3) - 1);
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kBK; kk += 4) {
      uint32_t a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const uint32_t*>(&qs[tm + 16 * i][kk]);
#pragma unroll
      for (int j = 0; j < 4; ++j) bb[j] = *reinterpret_cast<const uint32_t*>(&wsm[tn + 16 * j][kk]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = dp4a_ss(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
  const float sw = *reinterpret_cast<const float*>(packed + int64_t(N) * (K / 4));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm + 16 * i;
    if (m >= M) continue;
    const float sm = s[m];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn + 16 * j;
      if (n >= N) continue;
      y[int64_t(m) * N + n] = __fmul_rn(__fmul_rn(float(acc[i][j]), sm), sw);
      if (acc_out) acc_out[int64_t(m) * N + n] = acc[i][j];
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_gemm_i2s_int8_simt(const int8_t* q, const float* sc, const uint8_t* packed, int64_t M, int64_t N,
                                      int64_t K, float* y, int32_t* acc, cudaStream_t s) {
  dim3 grid(unsigned((N + kBN - 1) / kBN), unsigned((M + kBM - 1) / kBM));
  return launch(gemm_i2s_int8_simt_kernel, grid, dim3(256), 0, s, overlap_enabled(), q, sc, packed, int(M), int(N),
                int(K), y, acc);
}

}  // namespace bl
