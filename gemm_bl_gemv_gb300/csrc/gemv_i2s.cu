// i2_s GEMV, one token: y[n] = scale * sum_k w[n,k] x[k]
// ("Hesper/Layers/BitLinear", sections "i2_s Packing Format" and
// "BitLinear Mathematics").
//
// Decode.  A 32-bit word of a 128-element group holds bytes p..p+3 of the
// group; bits (7-2t):(6-2t) of byte p are the code of element 32t+p.  For
// the four shift classes we form byte masks of the codes:
//   class 0 (shift 0, elements 96+p): w & 0x03030303          -> code
//   class 1 (shift 2, elements 64+p): (w >> 2) & 0x03030303   -> code
//   class 2 (shift 4, elements 32+p): w & 0x30303030          -> 16*code
//   class 3 (shift 6, elements p)   : (w >> 2) & 0x30303030   -> 16*code
// and feed them to dp4a against activation digits.  Codes are c = w + 1, so
//   sum_k w_k X_k = sum_k c_k X_k - sum_k X_k,
// the second sum being the same for every row.
//
// Activations.  x is turned, once per CTA, into exact fixed-point integers
// X = rint(x * 2^F_c) with one exponent F_c per 128-element group c, chosen
// from the group's max|x| so that |X| < 2^(8D-2), and stored as D balanced
// int8 digits (X = sum_d digit_d 256^d).  D = 4 for fp32 input (30-bit
// magnitude: fp32 values within 6 binades of the group maximum are carried
// exactly, smaller ones with absolute error <= 2^-31 * group max), D = 3
// for bf16 input (exact within 14 binades).  Products and sums over a group
// are exact integers; the group sum is converted to fp32 once.
#include "bl_internal.h"
#include "gemv_tiled.cuh"

namespace bl {
namespace {

constexpr int kI2sR = 4;

template <int D, bool XB, bool YB>
struct I2sPolicy {
  static constexpr int kMaxThreads = 1024;
  struct Args {
    const uint8_t* packed;
    const void* x;
    void* y;
    int N, K;
  };
  // policy area: [xd: 8 steps x 4 classes x D x nC u32][sumx: D x nC][fexp: nC][cmax: nC][consts: 8]
  static __host__ __device__ uint32_t xd_words(int nC) { return 8u * 4u * D * nC; }
  static __host__ __device__ uint32_t bytes(int nC) { return (xd_words(nC) + D * nC + 2 * nC + 8) * 4; }

  static __device__ const uint8_t* weights(const Args& a) { return a.packed; }
  static __device__ const uint8_t* aux(const Args&) { return nullptr; }

  static __device__ float load_x(const Args& a, int e) {
    if (XB) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(a.x)[e]);
    return reinterpret_cast<const float*>(a.x)[e];
  }

  static __device__ void prepare(const Args& a, const TileGeom& g, uint8_t* smem, int tid, int T) {
    const int nC = g.nC;
    uint32_t* xd = reinterpret_cast<uint32_t*>(smem + g.off_pol);
    int* sumx = reinterpret_cast<int*>(xd + xd_words(nC));
    int* fexp = sumx + D * nC;
    int* cmax = fexp + nC;
    float* consts = reinterpret_cast<float*>(cmax + nC);
    for (int c = tid; c < nC; c += T) cmax[c] = 0;
    if (tid == 0) consts[1] = *reinterpret_cast<const float*>(a.packed + int64_t(a.N) * (a.K / 4));
    __syncthreads();
    // pass 1: max |x| of every 128-element group (non-negative floats order as ints)
    for (int qd = tid; qd < a.K / 4; qd += T) {
      float m = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) m = fmaxf(m, fabsf(load_x(a, 4 * qd + b)));
      atomicMax(&cmax[qd / 32], __float_as_int(m));
    }
    __syncthreads();
    for (int c = tid; c < nC; c += T) {
      const float m = __int_as_float(cmax[c]);
      int F = 0;
      if (m > 0.f) {
        int ex;
        frexpf(m, &ex);  // m < 2^ex
        F = (8 * D - 2) - ex;
      }
      fexp[c] = F;
    }
    __syncthreads();
    // pass 2: digits, in the rotated layout read by compute(): word
    // (step + c/4) % 8 of group c is read at step `step`, so that the 32
    // lanes of a warp (consecutive groups) hit 32 different banks.
    for (int qd = tid; qd < a.K / 4; qd += T) {
      const int e = qd * 4;
      const int c = e / 128;
      const int tt = (e % 128) / 32;
      const int sh = 3 - tt;
      const int w = (e % 32) / 4;
      const int step = (w - (c >> 2)) & 7;
      const int F = fexp[c];
      uint32_t dig[D];
#pragma unroll
      for (int d = 0; d < D; ++d) dig[d] = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        int X = __float2int_rn(ldexpf(load_x(a, e + b), F));
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const int v = ((X + 128) & 255) - 128;
          X = (X - v) >> 8;
          dig[d] |= uint32_t(v & 255) << (8 * b);
        }
      }
#pragma unroll
      for (int d = 0; d < D; ++d) xd[((step * 4 + sh) * D + d) * nC + c] = dig[d];
    }
    __syncthreads();
    // per-group digit sums (the sum_k X_k term)
    for (int idx = tid; idx < D * nC; idx += T) {
      const int d = idx / nC, c = idx % nC;
      int s = 0;
      for (int step = 0; step < 8; ++step)
        for (int sh = 0; sh < 4; ++sh) s = dp4a_us(0x01010101u, xd[((step * 4 + sh) * D + d) * nC + c], s);
      sumx[d * nC + c] = s;
    }
    __syncthreads();
  }

  static __device__ void compute(const Args& a, const TileGeom& g, const uint8_t* tile, const uint8_t* smem, int c,
                                 int grp, int row0, int rows, float* part) {
    const uint32_t* xd = reinterpret_cast<const uint32_t*>(smem + g.off_pol);
    const int* sumx = reinterpret_cast<const int*>(xd + xd_words(g.nC));
    const int nC = g.nC;
    const int64_t rb = g.row_bytes;
    const uint8_t* base = tile + int64_t(grp * kI2sR) * rb + 32 * c;
    int accA[kI2sR][D], accB[kI2sR][D];
#pragma unroll
    for (int r = 0; r < kI2sR; ++r)
#pragma unroll
      for (int d = 0; d < D; ++d) accA[r][d] = accB[r][d] = 0;
#pragma unroll 2
    for (int step = 0; step < 8; ++step) {
      const int w = (step + (c >> 2)) & 7;
      uint32_t xw[4][D];
#pragma unroll
      for (int sh = 0; sh < 4; ++sh)
#pragma unroll
        for (int d = 0; d < D; ++d) xw[sh][d] = xd[((step * 4 + sh) * D + d) * nC + c];
      uint32_t wd[kI2sR];
#pragma unroll
      for (int r = 0; r < kI2sR; ++r) wd[r] = *reinterpret_cast<const uint32_t*>(base + r * rb + 4 * w);
#pragma unroll
      for (int r = 0; r < kI2sR; ++r) {
        const uint32_t w2 = wd[r] >> 2;
        const uint32_t m0 = wd[r] & 0x03030303u, m1 = w2 & 0x03030303u;
        const uint32_t m2 = wd[r] & 0x30303030u, m3 = w2 & 0x30303030u;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          accA[r][d] = dp4a_us(m0, xw[0][d], accA[r][d]);
          accA[r][d] = dp4a_us(m1, xw[1][d], accA[r][d]);
          accB[r][d] = dp4a_us(m2, xw[2][d], accB[r][d]);
          accB[r][d] = dp4a_us(m3, xw[3][d], accB[r][d]);
        }
      }
    }
    // 2^-F_c as two normal factors (F_c may exceed the normal exponent range)
    const int F = sumx[D * nC + c];
    const float scA = ldexpf(1.f, -(F / 2)), scB = ldexpf(1.f, -(F - F / 2));
#pragma unroll
    for (int r = 0; r < kI2sR; ++r) {
      const int lr = grp * kI2sR + r;
      if (lr < rows) {
        float p = 0.f, sc = 1.f;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const int t = accA[r][d] + (accB[r][d] >> 4) - sumx[d * nC + c];
          p += float(t) * sc;
          sc *= 256.f;
        }
        part[lr * nC + c] = (p * scA) * scB;
      }
    }
  }

  static __device__ void finish(const Args& a, const TileGeom& g, const uint8_t* smem, const float* part, int row0,
                                int rows, int tid, int T) {
    const uint32_t* xd = reinterpret_cast<const uint32_t*>(smem + g.off_pol);
    const float* consts = reinterpret_cast<const float*>(xd + xd_words(g.nC) + D * g.nC + 2 * g.nC);
    const float s = consts[1];
    for (int r = tid; r < rows; r += T) {
      float acc = 0.f;
      const float* pr = part + r * g.nC;
      for (int c = 0; c < g.nC; ++c) acc += pr[c];
      const float yv = acc * s;
      if (YB)
        reinterpret_cast<uint16_t*>(a.y)[row0 + r] = f32_to_bf16_bits_rn(yv);
      else
        reinterpret_cast<float*>(a.y)[row0 + r] = yv;
    }
  }
};

template <int D, bool XB, bool YB>
cudaError_t run(const uint8_t* packed, const void* x, void* y, int64_t N, int64_t K, cudaStream_t st) {
  using Pol = I2sPolicy<D, XB, YB>;
  const int nC = int(K / 128);
  // threads = nC * P (<= 1024); aim for about 256 threads
  int P = 256 / nC;
  if (P < 1) P = 1;
  if (P > 8) P = 8;
  if (nC * P > 1024) return cudaErrorInvalidConfiguration;
  TileGeom g;
  int dev;
  cudaGetDevice(&dev);
  int max_optin = 0;
  cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // two CTAs per SM when possible
  const uint32_t budget = uint32_t(max_optin) / 2 - 2048;
  if (!plan_tiles(g, N, nC, P, kI2sR, 1, K / 4, 4, Pol::bytes(nC), budget) &&
      !plan_tiles(g, N, nC, P, kI2sR, 1, K / 4, 4, Pol::bytes(nC), uint32_t(max_optin)))
    return cudaErrorInvalidConfiguration;
  g.err = dev_error_ptr();
  auto kern = tiled_kernel<Pol>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(g.smem_bytes));
  if (e != cudaSuccess) return e;
  const int threads = (nC * P + 31) / 32 * 32;
  int blocks_per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kern, threads, g.smem_bytes);
  if (blocks_per_sm < 1) blocks_per_sm = 1;
  int grid = sm_count() * blocks_per_sm;
  if (grid > g.ntiles) grid = g.ntiles;
  typename Pol::Args a{packed, x, y, int(N), int(K)};
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(grid), dim3(threads), g.smem_bytes, st, pdl, a, g, pdl ? 1 : 0);
}

}  // namespace

cudaError_t launch_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                            int64_t K, cudaStream_t s) {
  const bool xb = xt == BL_BF16, yb = yt == BL_BF16;
  if (xb) return yb ? run<3, true, true>(packed, x, y, N, K, s) : run<3, true, false>(packed, x, y, N, K, s);
  return yb ? run<4, false, true>(packed, x, y, N, K, s) : run<4, false, false>(packed, x, y, N, K, s);
}

}  // namespace bl
