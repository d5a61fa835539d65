// W1A8 product, 1 <= M <= 8 tokens, "lane per row" kernel ("binary-gemm"
// card, sections "API" binary_gemm and "Method"):
//   dot[m,n,g] = sum_{k in g} w[n,k] q[m,k]                      (exact)
//   y[m,n]     = bf16( s[m] * sum_g ws[n,g] * dot[m,n,g] + bias[n] )
// using the card's identity dot(w, a) = 2 * sum_{b=1} a - sum a.
//
// A warp owns 16 rows.  Lane l works on the four rows l%4 + 4k (k < 4) and
// on every eighth scale group (phase l/4) of the warp's group range (split
// over `wk` warps when rows are few): each activation word read from shared
// memory serves four rows.  The eight phases of a row are added with three
// shuffles.  Each row's bits and scales for the range are bulk-copied into
// one shared-memory row slot whose stride is 32 bytes past a multiple of 128,
// so the 16-byte reads of every 8-lane phase (4 rows x 2 groups) hit
// distinct banks.  The activations of a group are rearranged once per CTA
// into per-bit-class words read by broadcast.
//
// Decode.  Element k of a 32-element word sits at bit k%32.  For bit class j
// (0..7) the mask  word & (0x01010101 << j)  holds the bits of elements j,
// j+8, j+16, j+24, one per byte (times 2^j), so one dp4a against the
// activation word of those four elements adds four products.  With one token
// the 8 class sums are kept apart and combined once per group
// (sum_j acc_j >> j); with more tokens the masks are shifted down once
// ((word >> j) & 0x01010101) and shared by all tokens.
//
// Used when K % 128 == 0, the group size is at most 256 and the number of
// groups per row is a multiple of 8 (every row slice and scale slice is then
// 16-byte aligned); other shapes take the tiled kernel in gemm_w1a8.cu.
//
// Fused activation quantization (XQ != 0).  The kernel can take the
// unquantized activations x (fp32 or bf16) instead of q and s: every CTA
// quantizes the <= 8 tokens itself, with the formula and the binary32
// operations of act_quant.cuh (per-token absmax, 127/amax, round to nearest
// even, clamp to +-127), so q and s are bit-identical to the stand-alone
// kernel's and the product is that of the two-launch sequence.
#pragma once
#include <algorithm>

#include "act_quant.cuh"
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kRows = 16;

struct Geom {
  int N, K, G, nG, wpc;  // rows, columns, group size, groups per row, words per group
  int wk, wr, stages, ntiles;
  int slot;              // bytes per row slot (bits then scales), odd multiple of 16
  int bits_bytes;        // bytes of bits in a slot (max over warps)
  uint32_t stage_bytes;
  uint32_t off_bar, off_stage, off_part, off_rec, off_qraw, smem;
  int rec_words;         // u32 per group record
  unsigned int* err;
};

// Per-token absmax int8 quantization (act_quant.cuh) of the MT tokens of
// x [MT, K] into qraw by the whole CTA (K % 8 == 0, x 16-byte aligned).
// Ends with a CTA barrier; qraw and scale are then valid for all threads.
template <int MT, bool XB>
__device__ __forceinline__ void quantize_tokens(const void* x, int K, int8_t* qraw, float* red, float* scale,
                                                float* inv) {
  token_scales<MT, XB>(x, K, red, scale, inv);
  const int n8 = K / 8;
  const size_t row_bytes = size_t(K) * (XB ? 2 : 4);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const void* xr = reinterpret_cast<const uint8_t*>(x) + m * row_bytes;
    const float iv = inv[m];
#pragma unroll 4
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
      float v[8];
      load8<XB>(xr, i, v);
      reinterpret_cast<uint2*>(qraw + size_t(m) * K)[i] = quant8(v, iv);
    }
  }
  __syncthreads();
}

// XQ: 0 = q and s given; 1 = fp32 x given; 2 = bf16 x given (quantized here)
template <int MT, bool DOTS, int XQ>
__global__ void __launch_bounds__((MT == 1 ? 512 : 256), (MT >= 2 && MT <= 4 ? 2 : 1)) gemm_w1a8_rows_kernel(const int8_t* __restrict__ q, const float* __restrict__ s,
                                                             const void* __restrict__ x,
                                                             const uint8_t* __restrict__ wq,
                                                             const uint8_t* __restrict__ ws,
                                                             const uint16_t* __restrict__ bias,
                                                             uint16_t* __restrict__ y, int32_t* __restrict__ dots,
                                                             Geom g, int early_weights) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int rt = warp / g.wk, ks = warp % g.wk;
  // group range of this warp, in units of 8 groups so every slice stays 16-byte aligned
  const int nu = g.nG / 8;
  const int c0 = 8 * (ks * nu / g.wk), c1 = 8 * ((ks + 1) * nu / g.wk);
  const int ngr = c1 - c0;
  const int r = lane & (kRows - 1), u = lane >> 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar) + warp * g.stages;
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + g.off_bar) + nwarps * g.stages;
  uint64_t* tbar = qbar + 1 + rt;
  uint8_t* ring = smem + g.off_stage + size_t(warp) * g.stages * g.stage_bytes;
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  uint32_t* rec = reinterpret_cast<uint32_t*>(smem + g.off_rec);
  int8_t* qraw = reinterpret_cast<int8_t*>(smem + g.off_qraw);
  __shared__ int abort_flag;
  __shared__ float tok_scale[MT], tok_inv[MT];
  __shared__ float red[32 * MT];

  const int tile_stride = int(gridDim.x) * g.wr;
  const int first = int(blockIdx.x) * g.wr + rt;
  const int my_tiles = first < g.ntiles ? (g.ntiles - 1 - first) / tile_stride + 1 : 0;
  const uint32_t bbytes = uint32_t(ngr) * uint32_t(g.G / 8);  // bits of the range per row
  const uint32_t sbytes = uint32_t(ngr) * 2;                   // scales of the range per row
  const int64_t row_bits = g.K / 8, row_sc = int64_t(g.nG) * 2;

  auto issue = [&](int i) {
    const int t = first + i * tile_stride;
    const int st = i % g.stages;
    const int row = t * kRows + r;
    const int nrows = min(kRows, g.N - t * kRows);
    if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(nrows) * (bbytes + sbytes));
    __syncwarp();
    if (row < g.N) {
      uint8_t* dst = ring + size_t(st) * g.stage_bytes + size_t(r) * g.slot;
      const uint64_t pol = policy_evict_first();
      if (u == 0)
        bulk_g2s(dst, wq + int64_t(row) * row_bits + int64_t(c0) * (g.G / 8), bbytes, &full[st], pol);
      else
        bulk_g2s(dst + g.bits_bytes, ws + int64_t(row) * row_sc + int64_t(c0) * 2, sbytes, &full[st], pol);
    }
  };

  if (lane == 0)
    for (int st = 0; st < g.stages; ++st) mbar_init(&full[st], 1);
  if (threadIdx.x == 0) {
    mbar_init(qbar, 1);
    for (int k = 0; k < g.wr; ++k) mbar_init(qbar + 1 + k, 32 * g.wk);
    abort_flag = 0;
  }
  fence_barrier_init();
  __syncthreads();
  const int npre = min(my_tiles, g.stages);
  if (early_weights)
    for (int i = 0; i < npre; ++i) issue(i);
  // let the next kernel's CTAs become resident now: they fetch their own
  // weights and then wait for this grid to complete before touching its outputs
  pdl_launch_dependents();
  pdl_wait();
  if (XQ == 0 && threadIdx.x == 0) {
    mbar_arrive_expect_tx(qbar, uint32_t(MT * g.K));
    bulk_g2s(qraw, q, uint32_t(MT * g.K), qbar, policy_evict_first());
  }
  if (!early_weights)
    for (int i = 0; i < npre; ++i) issue(i);
  if (XQ == 0) {
    if (!mbar_wait_bounded(qbar, 0, g.err)) abort_flag = 1;
  } else {
    quantize_tokens<MT, XQ == 2>(x, g.K, qraw, red, tok_scale, tok_inv);
  }
  const float* scale = XQ == 0 ? s : tok_scale;

  // group records: [word w][class j][token m] u32 holding q[m][G*c + 32w + j + 8b]
  // in byte b, then the per-token group sums of q
  for (int c = warp; c < g.nG; c += nwarps) {
    uint32_t* rc = rec + c * g.rec_words;
    int qs[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) qs[m] = 0;
    for (int e = lane; e < g.wpc * 8; e += 32) {
      const int w = e >> 3, j = e & 7;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int8_t* src = qraw + int64_t(m) * g.K + int64_t(g.G) * c + 32 * w + j;
        const uint32_t v = uint32_t(uint8_t(src[0])) | (uint32_t(uint8_t(src[8])) << 8) |
                           (uint32_t(uint8_t(src[16])) << 16) | (uint32_t(uint8_t(src[24])) << 24);
        rc[(w * 8 + j) * MT + m] = v;
        qs[m] = dp4a_us(0x01010101u, v, qs[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const int tot = redux_add(qs[m]);
      if (lane == 0) reinterpret_cast<int*>(rc)[g.wpc * 8 * MT + m] = tot;
    }
  }
  __syncthreads();

  const int a = lane & 3, v = lane >> 2;  // row slot, group phase
  for (int i = 0; i < my_tiles; ++i) {
    const int st = i % g.stages;
    const int t = first + i * tile_stride;
    if (!abort_flag && !mbar_wait_bounded(&full[st], uint32_t(i / g.stages) & 1u, g.err)) abort_flag = 1;
    __syncwarp();
    const uint8_t* buf = ring + size_t(st) * g.stage_bytes;
    float yacc[4][MT];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int m = 0; m < MT; ++m) yacc[k][m] = 0.f;
    for (int cc = v; cc < ngr; cc += 8) {
      const int c = c0 + cc;
      const uint32_t* rc = rec + c * g.rec_words;
      constexpr int NA = MT == 1 ? 8 : MT;
      int acc[4][NA];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int n = 0; n < NA; ++n) acc[k][n] = 0;
      // this group's words of the four rows (at most 8 words each: group <= 256)
      uint32_t wd[4][8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint8_t* gb = buf + size_t(a + 4 * k) * g.slot + cc * (g.G / 8);
        if ((g.wpc & 3) == 0) {
#pragma unroll
          for (int w0 = 0; w0 < 8; w0 += 4)
            if (w0 < g.wpc) {  // 16-byte reads: distinct banks per 8-lane phase
              const uint4 q4 = *reinterpret_cast<const uint4*>(gb + 4 * w0);
              wd[k][w0] = q4.x; wd[k][w0 + 1] = q4.y; wd[k][w0 + 2] = q4.z; wd[k][w0 + 3] = q4.w;
            }
        } else {
#pragma unroll
          for (int w = 0; w < 8; ++w)
            if (w < g.wpc) wd[k][w] = *reinterpret_cast<const uint32_t*>(gb + 4 * w);
        }
      }
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        if (w >= g.wpc) break;
        const uint32_t* qw = rc + w * 8 * MT;
        uint32_t q8[8];
        if (MT == 1) {  // one token: the word's eight class words by two 16-byte loads (records are 16-byte aligned)
          const uint4 a0 = *reinterpret_cast<const uint4*>(qw), a1 = *reinterpret_cast<const uint4*>(qw + 4);
          q8[0] = a0.x; q8[1] = a0.y; q8[2] = a0.z; q8[3] = a0.w;
          q8[4] = a1.x; q8[5] = a1.y; q8[6] = a1.z; q8[7] = a1.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t qj[MT];  // activation words of class j, one per token (broadcast reads)
#pragma unroll
          for (int m = 0; m < MT; ++m) qj[m] = MT == 1 ? q8[j] : 0u;
          if constexpr (MT > 1 && MT % 4 == 0) {
#pragma unroll
            for (int m4 = 0; m4 < MT; m4 += 4) {
              const uint4 v4 = *reinterpret_cast<const uint4*>(qw + j * MT + m4);
              qj[m4] = v4.x; qj[m4 + 1] = v4.y; qj[m4 + 2] = v4.z; qj[m4 + 3] = v4.w;
            }
          } else if constexpr (MT > 1 && MT % 2 == 0) {
#pragma unroll
            for (int m2 = 0; m2 < MT; m2 += 2) {
              const uint2 v2 = *reinterpret_cast<const uint2*>(qw + j * MT + m2);
              qj[m2] = v2.x; qj[m2 + 1] = v2.y;
            }
          } else if constexpr (MT > 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) qj[m] = qw[j * MT + m];
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (MT == 1) {
              acc[k][j] = dp4a_us(wd[k][w] & (0x01010101u << j), qj[0], acc[k][j]);
            } else {
              const uint32_t mk = (wd[k][w] >> j) & 0x01010101u;
#pragma unroll
              for (int m = 0; m < MT; ++m) acc[k][m] = dp4a_us(mk, qj[m], acc[k][m]);
            }
          }
        }
      }
      const int* qsum = reinterpret_cast<const int*>(rc + g.wpc * 8 * MT);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int row = t * kRows + a + 4 * k;
        const float wsf = __half2float(
            __ushort_as_half(*reinterpret_cast<const uint16_t*>(buf + size_t(a + 4 * k) * g.slot + g.bits_bytes + 2 * cc)));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          int S;
          if (MT == 1) {
            S = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) S += acc[k][j] >> j;
          } else {
            S = acc[k][m];
          }
          const int dot = 2 * S - qsum[m];
          if (DOTS && row < g.N) dots[(int64_t(m) * g.N + row) * g.nG + c] = dot;
          yacc[k][m] += wsf * float(dot);
        }
      }
    }
    // the eight phases of a row live in lanes a, a+4, ..., a+28 (same order on all)
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        yacc[k][m] += __shfl_xor_sync(0xffffffffu, yacc[k][m], 4);
        yacc[k][m] += __shfl_xor_sync(0xffffffffu, yacc[k][m], 8);
        yacc[k][m] += __shfl_xor_sync(0xffffffffu, yacc[k][m], 16);
      }
    __syncwarp();
    if (i + g.stages < my_tiles) issue(i + g.stages);
    if (g.wk == 1) {
      if (v == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = t * kRows + a + 4 * k;
          if (row < g.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              float val = yacc[k][m] * scale[m];
              if (bias) val += bf16_bits_to_f32(bias[row]);
              y[int64_t(m) * g.N + row] = f32_to_bf16_bits_rn(val);
            }
          }
        }
      }
    } else {
      float* pp = part + ((rt * 2 + (i & 1)) * g.wk) * kRows * MT;
      if (v == 0)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int m = 0; m < MT; ++m) pp[(ks * MT + m) * kRows + a + 4 * k] = yacc[k][m];
      mbar_arrive(tbar);
      if (!mbar_wait_bounded(tbar, uint32_t(i) & 1u, g.err)) abort_flag = 1;
      if (ks == 0 && v == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = t * kRows + a + 4 * k;
          if (row < g.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              float acc2 = 0.f;
              for (int kk = 0; kk < g.wk; ++kk) acc2 += pp[(kk * MT + m) * kRows + a + 4 * k];
              float val = acc2 * scale[m];
              if (bias) val += bf16_bits_to_f32(bias[row]);
              y[int64_t(m) * g.N + row] = f32_to_bf16_bits_rn(val);
            }
          }
        }
      }
    }
  }
  if (abort_flag && lane == 0) {
    for (int j = 0; j < my_tiles && j < g.stages; ++j) mbar_wait_bounded(&full[j], 0, nullptr);
    if (XQ == 0 && warp == 0) mbar_wait_bounded(qbar, 0, nullptr);
  }
}

bool plan(Geom& g, int M, int64_t N, int64_t K, int G, int max_smem, int nsm) {
  // up to 16 warps per CTA for one token (more warps hide the decode's
  // dependency chains; the ring then holds fewer stages per warp), else 8
  const int max_warps = M == 1 ? 16 : 8;
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.N = int(N);
  g.K = int(K);
  g.G = G;
  g.nG = int(K / G);
  g.wpc = G / 32;
  g.ntiles = int((N + kRows - 1) / kRows);
  const int nu = g.nG / 8;
  int wk = 1;
  while (wk < 8 && wk < nu && int64_t(g.ntiles) * wk < int64_t(max_warps) * nsm) ++wk;
  g.wk = wk;
  int wr = std::max(1, max_warps / wk);
  while (wr > 1 && (g.ntiles + wr - 1) / wr < nsm) --wr;
  g.wr = wr;
  const int max_units = (nu + wk - 1) / wk;
  g.bits_bytes = int(max_units * 8 * (G / 8));
  // slot = 32 (mod 128): (row slot a, group phase v) pairs of an 8-lane phase map to distinct 16-byte units
  int slot = int(up(uint64_t(g.bits_bytes) + max_units * 8 * 2, 16));
  while (slot % 128 != 32) slot += 16;
  g.slot = slot;
  g.stage_bytes = uint32_t(up(uint64_t(kRows) * slot, 128));
  g.rec_words = int(up(uint64_t(g.wpc) * 8 * M + M, 4));  // 16-byte records,
  if ((g.rec_words / 4) % 2 == 0) g.rec_words += 4;          // an odd number of 16-byte units apart
  const int warps = g.wk * g.wr;
  const int64_t tiles_per_warp = (g.ntiles + int64_t(g.wr) * nsm - 1) / (int64_t(g.wr) * nsm);
  for (int st = int(std::min<int64_t>(4, std::max<int64_t>(1, tiles_per_warp))); st >= 1; --st) {
    uint64_t off = 0;
    g.off_bar = uint32_t(off);
    off = up(off + 8ull * (warps * st + 1 + g.wr), 128);
    g.off_stage = uint32_t(off);
    off = up(off + uint64_t(warps) * st * g.stage_bytes, 128);
    g.off_part = uint32_t(off);
    off = up(off + (g.wk > 1 ? 4ull * g.wr * 2 * g.wk * kRows * M : 0), 128);
    g.off_rec = uint32_t(off);
    off = up(off + 4ull * g.nG * g.rec_words, 128);
    g.off_qraw = uint32_t(off);
    off = up(off + uint64_t(M) * K, 128);
    if (off <= uint64_t(max_smem)) {
      g.stages = st;
      g.smem = uint32_t(off);
      return true;
    }
  }
  return false;
}

struct Plan {
  Geom g;
  int grid, threads;
};

template <int MT, bool DOTS, int XQ>
cudaError_t run(const int8_t* q, const float* s, const void* x, const int32_t* wq, const uint16_t* ws,
                const uint16_t* bias, int64_t N, int64_t K, int G, uint16_t* y, int32_t* dots, cudaStream_t st) {
  auto kern = gemm_w1a8_rows_kernel<MT, DOTS, XQ>;
  static PlanCache<Plan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  Plan p{};
  if (!cache.get(dev, N, K * 4096 + G, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int nsm = sm_count();
    // the kernel's static shared memory (the token scales of the fused
    // quantization among it) comes out of the same per-block budget
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    const int budget = max_optin - int(fa.sharedSizeBytes);
    if (!plan(p.g, MT, N, K, G, budget, nsm)) return cudaErrorNotSupported;
    e = raise_smem_cap(kern, dev, budget);
    if (e != cudaSuccess) return e;
    p.threads = 32 * p.g.wk * p.g.wr;
    int bps = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, p.threads, p.g.smem);
    if (bps < 1) bps = 1;
    p.grid = (p.g.ntiles + p.g.wr - 1) / p.g.wr;
    if (p.grid > nsm * bps) p.grid = nsm * bps;
    p.g.err = dev_error_ptr();
    cache.put(dev, N, K * 4096 + G, p);
  }
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(p.grid), dim3(p.threads), p.g.smem, st, pdl, q, s, x,
                reinterpret_cast<const uint8_t*>(wq), reinterpret_cast<const uint8_t*>(ws), bias, y, dots, p.g,
                pdl ? 1 : 0);
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
}  // namespace bl
