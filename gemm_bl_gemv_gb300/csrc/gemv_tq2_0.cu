// TQ2_0 GEMV, one token ("Hesper/Quantization/TQ2_0", section "TQ2_0 Format"):
//   y[n] = sum_b d[n,b] * sum_{j<256} w[n,256b+j] x[256b+j]
// A block is 64 code bytes then its fp16 scale: 66 bytes, so blocks of odd
// index inside a tile start 2 bytes past a 4-byte boundary; their code words
// are assembled from two aligned shared-memory words with a funnel shift.
//
// Decode.  Element j of a block sits in byte j/4 at shift 2*(j%4) with codes
// 00 -> 0, 01 -> +1, 11 -> -1.  XOR with 0b01 maps the codes to
// t = 1 - w in {1, 0, 2}, so sum_j w_j X_j = sum_j X_j - sum_j t_j X_j and
// the same byte-mask + dp4a decode as i2_s applies (classes = shift 0,2,4,6,
// i.e. elements 16i+4b+{0,1,2,3} of word i, byte b).  The per-block integer
// sum is converted to fp32 once and multiplied by the block scale.
//
// Activations: exact fixed-point digits as in the i2_s GEMV, with one
// exponent per 256-element block (D = 4 for fp32 x, D = 3 for bf16 x).
#include "bl_internal.h"
#include "gemv_tiled.cuh"

namespace bl {
namespace {

constexpr int kTqR = 4;

template <int D, bool XB>
struct Tq2Policy {
  static constexpr int kMaxThreads = 1024;
  struct Args {
    const uint8_t* packed;
    const void* x;
    float* y;
    int N, K;
  };
  // policy area: [xd: 16 words x 4 classes x D x nC u32][sumx: D x nC][fexp: nC][cmax: nC]
  static __host__ __device__ uint32_t xd_words(int nC) { return 16u * 4u * D * nC; }
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
    for (int c = tid; c < nC; c += T) cmax[c] = 0;
    __syncthreads();
    for (int idx = tid; idx < nC * 16; idx += T) {
      float m = 0.f;
      for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(load_x(a, 16 * idx + j)));
      atomicMax(&cmax[idx / 16], __float_as_int(m));
    }
    __syncthreads();
    for (int c = tid; c < nC; c += T) {
      const float m = __int_as_float(cmax[c]);
      int F = 0;
      if (m > 0.f) {
        int ex;
        frexpf(m, &ex);
        F = (8 * D - 2) - ex;
      }
      fexp[c] = F;
    }
    __syncthreads();
    // one (block c, word i) per iteration: elements 256c + 16i + 0..15
    for (int idx = tid; idx < nC * 16; idx += T) {
      const int c = idx / 16, i = idx % 16;
      const int F = fexp[c];
      uint32_t dig[4][D];
#pragma unroll
      for (int sh = 0; sh < 4; ++sh)
#pragma unroll
        for (int d = 0; d < D; ++d) dig[sh][d] = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        int X = __float2int_rn(ldexpf(load_x(a, 256 * c + 16 * i + j), F));
        const int b = j >> 2, sh = j & 3;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const int v = ((X + 128) & 255) - 128;
          X = (X - v) >> 8;
          dig[sh][d] |= uint32_t(v & 255) << (8 * b);
        }
      }
#pragma unroll
      for (int sh = 0; sh < 4; ++sh)
#pragma unroll
        for (int d = 0; d < D; ++d) xd[((i * 4 + sh) * D + d) * nC + c] = dig[sh][d];
    }
    __syncthreads();
    for (int idx = tid; idx < D * nC; idx += T) {
      const int d = idx / nC, c = idx % nC;
      int s = 0;
      for (int i = 0; i < 16; ++i)
        for (int sh = 0; sh < 4; ++sh) s = dp4a_us(0x01010101u, xd[((i * 4 + sh) * D + d) * nC + c], s);
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
    int accA[kTqR][D], accB[kTqR][D];
#pragma unroll
    for (int r = 0; r < kTqR; ++r)
#pragma unroll
      for (int d = 0; d < D; ++d) accA[r][d] = accB[r][d] = 0;
    // byte offset of block c of row (grp*R + r) inside the tile
    uint32_t boff[kTqR];
#pragma unroll
    for (int r = 0; r < kTqR; ++r) boff[r] = uint32_t((grp * kTqR + r) * rb + 66 * c);
#pragma unroll 2
    for (int i = 0; i < 16; ++i) {
      uint32_t xw[4][D];
#pragma unroll
      for (int sh = 0; sh < 4; ++sh)
#pragma unroll
        for (int d = 0; d < D; ++d) xw[sh][d] = xd[((i * 4 + sh) * D + d) * nC + c];
#pragma unroll
      for (int r = 0; r < kTqR; ++r) {
        const uint32_t addr = boff[r] + 4 * i;
        const uint32_t* p = reinterpret_cast<const uint32_t*>(tile + (addr & ~3u));
        const uint32_t wd = __funnelshift_r(p[0], p[1], (addr & 3u) * 8) ^ 0x55555555u;
        const uint32_t w2 = wd >> 2;
        const uint32_t m0 = wd & 0x03030303u, m1 = w2 & 0x03030303u;
        const uint32_t m2 = wd & 0x30303030u, m3 = w2 & 0x30303030u;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          accA[r][d] = dp4a_us(m0, xw[0][d], accA[r][d]);
          accA[r][d] = dp4a_us(m1, xw[1][d], accA[r][d]);
          accB[r][d] = dp4a_us(m2, xw[2][d], accB[r][d]);
          accB[r][d] = dp4a_us(m3, xw[3][d], accB[r][d]);
        }
      }
    }
    const int F = sumx[D * nC + c];
    const float scA = ldexpf(1.f, -(F / 2)), scB = ldexpf(1.f, -(F - F / 2));
#pragma unroll
    for (int r = 0; r < kTqR; ++r) {
      const int lr = grp * kTqR + r;
      if (lr < rows) {
        float p = 0.f, sc = 1.f;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const int t = sumx[d * nC + c] - (accA[r][d] + (accB[r][d] >> 4));
          p += float(t) * sc;
          sc *= 256.f;
        }
        const uint16_t dbits = *reinterpret_cast<const uint16_t*>(tile + boff[r] + 64);
        part[lr * nC + c] = __half2float(__ushort_as_half(dbits)) * ((p * scA) * scB);
      }
    }
  }

  static __device__ void finish(const Args& a, const TileGeom& g, const uint8_t* smem, const float* part, int row0,
                                int rows, int tid, int T) {
    for (int r = tid; r < rows; r += T) {
      float acc = 0.f;
      const float* pr = part + r * g.nC;
      for (int c = 0; c < g.nC; ++c) acc += pr[c];
      a.y[row0 + r] = acc;
    }
  }
};

template <int D, bool XB>
cudaError_t run(const uint8_t* packed, const void* x, float* y, int64_t N, int64_t K, cudaStream_t st) {
  using Pol = Tq2Policy<D, XB>;
  const int nC = int(K / 256);
  int P = 256 / nC;
  if (P < 1) P = 1;
  if (P > 8) P = 8;
  // tile bytes must be a multiple of 16 for the bulk copy: TR * nC * 66 % 16 == 0
  while ((P * kTqR * nC * 66) % 16 != 0) ++P;
  if (nC * P > 1024) return cudaErrorInvalidConfiguration;
  TileGeom g;
  int dev;
  cudaGetDevice(&dev);
  int max_optin = 0;
  cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const uint32_t budget = uint32_t(max_optin) / 2 - 2048;
  if (!plan_tiles(g, N, nC, P, kTqR, 1, int64_t(nC) * 66, 4, Pol::bytes(nC), budget) &&
      !plan_tiles(g, N, nC, P, kTqR, 1, int64_t(nC) * 66, 4, Pol::bytes(nC), uint32_t(max_optin)))
    return cudaErrorInvalidConfiguration;
  g.err = dev_error_ptr();
  auto kern = tiled_kernel<Pol>;
  cudaError_t e = raise_smem_cap(kern, dev, max_optin);
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

cudaError_t launch_gemv_tq2_0(const uint8_t* packed, const void* x, bl_dtype xt, float* y, int64_t N, int64_t K,
                              cudaStream_t s) {
  if (xt == BL_BF16) return run<3, true>(packed, x, y, N, K, s);
  return run<4, false>(packed, x, y, N, K, s);
}

}  // namespace bl
