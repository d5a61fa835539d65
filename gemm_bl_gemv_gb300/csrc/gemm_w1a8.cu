// W1A8 product for 1 <= M <= 8 tokens, tiled kernel for shapes the
// lane-per-row kernel (gemm_w1a8_rows.cuh) does not take ("binary-gemm"
// card, sections "API" binary_gemm and "Method"):
//   dot[m,n,g] = sum_{k in g} w[n,k] q[m,k]     (exact)
//   y[m,n]     = bf16( s[m] * sum_g ws[n,g] * dot[m,n,g] + bias[n] )
// with the card's identity dot(w, a) = 2 * sum_{b=1} a - sum a (stored bit
// b = (w+1)/2), so only the set bits are multiplied.
//
// Decode.  Element k of a 32-element word sits at bit k%32.  For bit class j
// (0..7) the byte mask  word & (0x01010101 << j)  (or (word >> j) & 0x01010101)
// holds the bits of elements j, j+8, j+16, j+24, one per byte, so one dp4a
// against the int8 activations of those four elements adds four products.
// With M = 1 the unshifted masks are used and the 8 class sums are combined
// once per group (sum_j acc_j >> j); with M > 1 the masks are shifted once
// and shared by all tokens.
//
// A chunk of the tiled skeleton is one scale group (group/32 words); the
// group scales of the tile's rows travel in the same bulk copy as the bits.
//
// XQ != 0: the kernel takes unquantized activations (1 = fp32, 2 = bf16) and
// quantizes them per token in its prologue with the helpers of act_quant.cuh,
// so the codes and scales are those of the stand-alone kernel.
#include "act_quant.cuh"
#include "bl_internal.h"
#include "gemv_tiled.cuh"

namespace bl {
namespace {

constexpr int kW1R = 4;

template <int MT, bool DOTS, int XQ>
struct W1a8Policy {
  static constexpr int kMaxThreads = 1024;
  struct Args {
    const int8_t* q;
    const float* s;
    const void* x;  // XQ != 0: [MT, K] activations to quantize
    const int32_t* wq;
    const uint16_t* ws;
    const uint16_t* bias;
    uint16_t* y;
    int32_t* dots;
    int N, K, G;
  };
  // policy area: [qd: MT x WPC x 8 x nC u32][qsum: MT x nC int][8 spare]
  //              [XQ: reduction 32 x MT, scale MT, inv MT floats]
  static __host__ __device__ uint32_t qd_words(int nC, int wpc) { return uint32_t(MT) * wpc * 8u * nC; }
  static __host__ __device__ uint32_t tq_word(int nC, int wpc) { return qd_words(nC, wpc) + MT * nC + 8; }
  static __host__ __device__ uint32_t bytes(int nC, int wpc) {
    return (tq_word(nC, wpc) + (XQ ? 34 * MT : 0)) * 4;
  }

  static __device__ const uint8_t* weights(const Args& a) { return reinterpret_cast<const uint8_t*>(a.wq); }
  static __device__ const uint8_t* aux(const Args& a) { return reinterpret_cast<const uint8_t*>(a.ws); }

  // rotation of the word order inside a group so that the lanes of a warp,
  // which read consecutive groups, read 32 different banks
  static __device__ __forceinline__ int rot(int c, int wpc) { return wpc < 32 ? (c / (32 / wpc)) % wpc : 0; }

  static __device__ void prepare(const Args& a, const TileGeom& g, uint8_t* smem, int tid, int T) {
    uint32_t* qd = reinterpret_cast<uint32_t*>(smem + g.off_pol);
    const int nC = g.nC, wpc = a.G / 32;
    int* qsum = reinterpret_cast<int*>(qd + qd_words(nC, wpc));
    float* tq = reinterpret_cast<float*>(qd + tq_word(nC, wpc));
    if (XQ) token_scales<MT, XQ == 2>(a.x, a.K, tq, tq + 32 * MT, tq + 33 * MT);
    // one (token m, group c, word w) per iteration: elements G*c + 32w + 0..31
    for (int idx = tid; idx < MT * nC * wpc; idx += T) {
      const int m = idx / (nC * wpc);
      const int c = (idx / wpc) % nC;
      const int w = idx % wpc;
      const int64_t e0 = int64_t(m) * a.K + int64_t(a.G) * c + 32 * w;
      uint32_t v[8];
      if (XQ) {
        const float inv = tq[33 * MT + m];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float f[8];
          load8<XQ == 2>(a.x, e0 / 8 + k, f);
          const uint2 b = quant8(f, inv);
          v[2 * k] = b.x;
          v[2 * k + 1] = b.y;
        }
      } else {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.q + e0);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = src[k];
      }
      const int step = (w - rot(c, wpc) + wpc) % wpc;
      // class j collects bytes j, j+8, j+16, j+24 of the 32 activation bytes
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sh = 8 * (j & 3), hi = j >> 2;
        const uint32_t b0 = (v[0 + hi] >> sh) & 0xFF, b1 = (v[2 + hi] >> sh) & 0xFF;
        const uint32_t b2 = (v[4 + hi] >> sh) & 0xFF, b3 = (v[6 + hi] >> sh) & 0xFF;
        qd[((m * wpc + step) * 8 + j) * nC + c] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < MT * nC; idx += T) {
      const int m = idx / nC, c = idx % nC;
      int s = 0;
      for (int st = 0; st < wpc; ++st)
        for (int j = 0; j < 8; ++j) s = dp4a_us(0x01010101u, qd[((m * wpc + st) * 8 + j) * nC + c], s);
      qsum[m * nC + c] = s;
    }
    __syncthreads();
  }

  static __device__ void compute(const Args& a, const TileGeom& g, const uint8_t* tile, const uint8_t* smem, int c,
                                 int grp, int row0, int rows, float* part) {
    const int nC = g.nC, wpc = a.G / 32;
    const uint32_t* qd = reinterpret_cast<const uint32_t*>(smem + g.off_pol);
    const int* qsum = reinterpret_cast<const int*>(qd + qd_words(nC, wpc));
    const int64_t rb = g.row_bytes;
    const uint8_t* base = tile + int64_t(grp * kW1R) * rb + int64_t(a.G / 8) * c;
    const int r0 = rot(c, wpc);
    constexpr int NA = (MT == 1) ? 8 : MT;
    int acc[kW1R][NA];
#pragma unroll
    for (int r = 0; r < kW1R; ++r)
#pragma unroll
      for (int k = 0; k < NA; ++k) acc[r][k] = 0;
    for (int step = 0; step < wpc; ++step) {
      int w = step + r0;
      if (w >= wpc) w -= wpc;
      uint32_t wd[kW1R];
#pragma unroll
      for (int r = 0; r < kW1R; ++r) wd[r] = *reinterpret_cast<const uint32_t*>(base + r * rb + 4 * w);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t qw[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) qw[m] = qd[((m * wpc + step) * 8 + j) * nC + c];
#pragma unroll
        for (int r = 0; r < kW1R; ++r) {
          if (MT == 1) {
            acc[r][j] = dp4a_us(wd[r] & (0x01010101u << j), qw[0], acc[r][j]);
          } else {
            const uint32_t mk = (wd[r] >> j) & 0x01010101u;
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = dp4a_us(mk, qw[m], acc[r][m]);
          }
        }
      }
    }
    const int nG = nC;
#pragma unroll
    for (int r = 0; r < kW1R; ++r) {
      const int lr = grp * kW1R + r;
      if (lr < rows) {
        const uint16_t wsb = *reinterpret_cast<const uint16_t*>(tile + g.aux_off + (int64_t(lr) * nG + c) * 2);
        const float wsf = __half2float(__ushort_as_half(wsb));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          int S;
          if (MT == 1) {
            S = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) S += acc[r][j] >> j;
          } else {
            S = acc[r][m];
          }
          const int dot = 2 * S - qsum[m * nC + c];
          if (DOTS) a.dots[(int64_t(m) * a.N + row0 + lr) * nG + c] = dot;
          part[(m * g.TR + lr) * nC + c] = wsf * float(dot);
        }
      }
    }
  }

  static __device__ void finish(const Args& a, const TileGeom& g, const uint8_t* smem, const float* part, int row0,
                                int rows, int tid, int T) {
    for (int o = tid; o < MT * rows; o += T) {
      const int m = o / rows, r = o % rows;
      const float* pr = part + (m * g.TR + r) * g.nC;
      float acc = 0.f;
      for (int c = 0; c < g.nC; ++c) acc += pr[c];
      const float sm = XQ ? reinterpret_cast<const float*>(
                                reinterpret_cast<const uint32_t*>(smem + g.off_pol) + tq_word(g.nC, a.G / 32))[32 * MT + m]
                          : a.s[m];
      float yv = acc * sm;
      if (a.bias) yv += bf16_bits_to_f32(a.bias[row0 + r]);
      a.y[int64_t(m) * a.N + row0 + r] = f32_to_bf16_bits_rn(yv);
    }
  }
};

template <int MT, bool DOTS, int XQ>
cudaError_t run(const int8_t* q, const float* s, const void* x, const int32_t* wq, const uint16_t* ws,
                const uint16_t* bias, int64_t N, int64_t K, int G, uint16_t* y, int32_t* dots, cudaStream_t st) {
  using Pol = W1a8Policy<MT, DOTS, XQ>;
  const int nC = int(K / G), wpc = G / 32;
  int P = 256 / nC;
  if (P < 1) P = 1;
  if (P > 8) P = 8;
  // the scale segment of a tile must be a multiple of 16 bytes: TR * nC * 2 % 16 == 0
  while ((P * kW1R * nC * 2) % 16 != 0) ++P;
  if (nC * P > 1024) return cudaErrorInvalidConfiguration;
  TileGeom g;
  int dev;
  cudaGetDevice(&dev);
  int max_optin = 0;
  cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const uint32_t budget = uint32_t(max_optin) / 2 - 2048;
  const uint32_t pb = Pol::bytes(nC, wpc);
  if (!plan_tiles(g, N, nC, P, kW1R, MT, K / 8, 4, pb, budget, int64_t(nC) * 2) &&
      !plan_tiles(g, N, nC, P, kW1R, MT, K / 8, 4, pb, uint32_t(max_optin), int64_t(nC) * 2))
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
  typename Pol::Args a{q, s, x, wq, ws, bias, y, dots, int(N), int(K), G};
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(grid), dim3(threads), g.smem_bytes, st, pdl, a, g, pdl ? 1 : 0);
}

template <bool DOTS, int XQ>
cudaError_t dispatch(int M, const int8_t* q, const float* s, const void* x, const int32_t* wq, const uint16_t* ws,
                     const uint16_t* bias, int64_t N, int64_t K, int G, uint16_t* y, int32_t* dots, cudaStream_t st) {
  switch (M) {
    case 1: return run<1, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 2: return run<2, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 3: return run<3, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 4: return run<4, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 5: return run<5, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 6: return run<6, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 7: return run<7, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
    case 8: return run<8, DOTS, XQ>(q, s, x, wq, ws, bias, N, K, G, y, dots, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm_w1a8(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws,
                             const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                             int32_t* dots, cudaStream_t st) {
  if (M > 8) {
    if (dots || !w1a8_tc_applicable(M, K, group)) return cudaErrorNotSupported;
    return launch_gemm_w1a8_tc(q, s, wq, ws, bias, M, N, K, group, y, st);
  }
  if (w1a8_m1_applicable(M, N, K, group)) {
    const cudaError_t e = launch_gemm_w1a8_m1(q, s, nullptr, BL_F32, wq, ws, bias, N, K, y, dots, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (w1a8_rows_applicable(M, K, group)) {
    const cudaError_t e = launch_gemm_w1a8_rows(q, s, wq, ws, bias, M, N, K, group, y, dots, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (dots) return dispatch<true, 0>(int(M), q, s, nullptr, wq, ws, bias, N, K, group, y, dots, st);
  return dispatch<false, 0>(int(M), q, s, nullptr, wq, ws, bias, N, K, group, y, dots, st);
}

cudaError_t launch_gemm_w1a8_act_tiled(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws,
                                       const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                       cudaStream_t st) {
  if (xt == BL_BF16) return dispatch<false, 2>(int(M), nullptr, nullptr, x, wq, ws, bias, N, K, group, y, nullptr, st);
  return dispatch<false, 1>(int(M), nullptr, nullptr, x, wq, ws, bias, N, K, group, y, nullptr, st);
}

}  // namespace bl
