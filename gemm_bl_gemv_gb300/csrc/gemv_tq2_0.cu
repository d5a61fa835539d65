// TQ2_0 GEMV, one token ("Hesper/Quantization/TQ2_0", section "TQ2_0 Format"):
//   y[n] = sum_b d[n,b] * sum_{j<256} w[n,256b+j] x[256b+j]
//
// Work decomposition.  A warp owns a tile of 8 consecutive rows; four lanes
// work on each row and take every fourth 256-element block; their sums are
// added with two shuffles.  The grid has one CTA per SM and CTA b takes the
// contiguous tile range [b T / G, (b + 1) T / G), so every SM decodes the
// same number of tiles (to one), its warps taking them in turn.  A tile is contiguous in memory (8 * 66 bytes per
// block, always a multiple of 16), so one thread bulk-copies it
// (cp.async.bulk) into a ring buffer of the warp.  Blocks of odd index start
// 2 bytes past a 4-byte boundary; their code words are assembled from two
// aligned shared-memory words with a funnel shift.
//
// Decode.  Element j of a block sits in byte j/4 at shift 2*(j%4) with codes
// 00 -> 0, 01 -> +1, 11 -> -1.  XOR with 0b01 maps the codes to
// t = 1 - w in {1, 0, 2}, so sum_j w_j X_j = sum_j X_j - sum_j t_j X_j and a
// byte-mask + dp4a decode applies: in word i of a block, byte b holds
// elements 16i+4b+{0,1,2,3} at shifts 0,2,4,6:
//   shift 0: w & 0x03030303, shift 2: (w >> 2) & 0x03030303,
//   shift 4: w & 0x30303030 (x16), shift 6: (w >> 2) & 0x30303030 (x16).
// The per-block integer sum is converted to fp32 once and multiplied by the
// block scale.
//
// Activations: once per CTA, exact fixed-point integers with one exponent per
// 256-element block (as in the i2_s GEMV: D = 4 bytes for fp32 x, D = 3 for
// bf16 x, two's complement, signed top byte), read by broadcast.
#include <algorithm>

#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kRows = 8;  // rows per warp tile (four lanes per row)

struct Geom {
  int N, K, nb;          // rows, columns, 256-element blocks per row
  int wpb, stages, ntiles;
  int64_t row_bytes;     // nb * 66
  uint32_t stage_bytes;  // kRows * row_bytes (+4) rounded up to 128
  uint32_t off_bar, off_stage, off_rec, off_xraw, smem;
  int xbytes;
  unsigned int* err;
};

// Per-block activation record: [16 words][4 shifts][D] u32, D digit sums,
// two fp32 factors whose product is 2^-F_b, padding to 16 bytes.
template <int D>
struct Rec {
  static constexpr int kWords = (64 * D + D + 2 + 3) / 4 * 4;
};

template <int D, bool XB>
__device__ __forceinline__ void prepare_x(const uint8_t* xraw, int nb, uint32_t* xrec, int warp, int nwarps,
                                          int lane) {
  constexpr int RW = Rec<D>::kWords;
  for (int c = warp; c < nb; c += nwarps) {
    // lane l holds elements 8l..8l+7 of block c: word i = l/2, bytes 2(l&1), 2(l&1)+1
    float v[8];
    const int e0 = c * 256 + 8 * lane;
    if (XB) {
      const uint4 q = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(xraw) + e0);
      const uint32_t h[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(h[k] << 16);
        v[2 * k + 1] = __uint_as_float(h[k] & 0xFFFF0000u);
      }
    } else {
      const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xraw) + e0);
      const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xraw) + e0 + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    float mm = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) mm = fmaxf(mm, fabsf(v[k]));
    const float m = __uint_as_float(redux_max_u32(__float_as_uint(mm)));
    const int F = m > 0.f ? (8 * D - 1) - exponent_of(m) : 0;
    const int fa = F / 2, fb = F - fa;
    const float sA = exp2i(fa), sB = exp2i(fb);
    int X[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      constexpr int kLim = int((1u << (8 * D - 1)) - 1u);
      X[k] = max(-kLim, min(kLim, __float2int_rn(__fmul_rn(__fmul_rn(v[k], sA), sB))));
    }
    uint32_t* rec = xrec + c * RW;
    const int i = lane >> 1, half = lane & 1;
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const uint32_t sel = uint32_t(d) | (uint32_t(d + 4) << 4);
      int dsum = 0;
#pragma unroll
      for (int sh = 0; sh < 4; ++sh) {
        // this lane's two bytes of word i, shift class sh: elements 8*half+sh and 8*half+4+sh
        const uint32_t mine = __byte_perm(uint32_t(X[sh]), uint32_t(X[4 + sh]), sel);  // low half used
        const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
        const uint32_t word = half ? __byte_perm(other, mine, 0x5410) : __byte_perm(mine, other, 0x5410);
        if (half == 0) rec[(i * 4 + sh) * D + d] = word;
        dsum = (d == D - 1) ? dp4a_us(0x00000101u, mine, dsum) : dp4a_uu(0x00000101u, mine, dsum);
      }
      const int s = redux_add(dsum);
      if (lane == 0) reinterpret_cast<int*>(rec)[64 * D + d] = s;
    }
    if (lane == 0) {
      reinterpret_cast<float*>(rec)[64 * D + D] = exp2i(-fa);
      reinterpret_cast<float*>(rec)[64 * D + D + 1] = exp2i(-fb);
    }
  }
}

template <int D, bool XB>
__global__ void __launch_bounds__(512) gemv_tq2_0_kernel(const uint8_t* __restrict__ packed,
                                                         const void* __restrict__ x, float* __restrict__ y, Geom g,
                                                         int early_weights) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RW = Rec<D>::kWords;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int r = lane & (kRows - 1), v = lane >> 3;  // row of the tile, block residue
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar) + warp * g.stages;
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + g.off_bar) + nwarps * g.stages;
  uint8_t* ring = smem + g.off_stage + size_t(warp) * g.stages * g.stage_bytes;
  uint32_t* xrec = reinterpret_cast<uint32_t*>(smem + g.off_rec);
  uint8_t* xraw = smem + g.off_xraw;
  __shared__ int abort_flag;

  const int t0 = int(int64_t(blockIdx.x) * g.ntiles / gridDim.x);
  const int t1 = int(int64_t(blockIdx.x + 1) * g.ntiles / gridDim.x);
  const int tile_stride = nwarps;
  const int first = t0 + warp;
  const int my_tiles = first < t1 ? (t1 - 1 - first) / tile_stride + 1 : 0;

  auto issue = [&](int i) {  // lane 0 only
    const int t = first + i * tile_stride;
    const int st = i % g.stages;
    const int nrows = min(kRows, g.N - t * kRows);
    const uint64_t bytes = uint64_t(nrows) * uint64_t(g.row_bytes);
    const uint32_t b16 = uint32_t(bytes & ~uint64_t(15));
    uint8_t* dst = ring + size_t(st) * g.stage_bytes;
    const uint8_t* src = packed + int64_t(t) * kRows * g.row_bytes;
    // a last tile that is not a multiple of 16 bytes: its tail goes by plain loads
    for (uint32_t k = b16; k < uint32_t(bytes); ++k) dst[k] = src[k];
    mbar_arrive_expect_tx(&full[st], b16);
    if (b16) bulk_g2s(dst, src, b16, &full[st], policy_evict_first());
  };

  if (lane == 0)
    for (int st = 0; st < g.stages; ++st) mbar_init(&full[st], 1);
  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    abort_flag = 0;
  }
  fence_barrier_init();
  __syncthreads();
  const int npre = min(my_tiles, g.stages);
  if (early_weights && lane == 0)
    for (int i = 0; i < npre; ++i) issue(i);
  // let the next kernel's CTAs become resident now: they fetch their own
  // weights and then wait for this grid to complete before touching its outputs
  pdl_launch_dependents();
  pdl_wait();
  const bool x_bulk = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  if (threadIdx.x == 0 && x_bulk) {
    mbar_arrive_expect_tx(xbar, uint32_t(g.xbytes));
    bulk_g2s(xraw, x, uint32_t(g.xbytes), xbar, policy_evict_first());
  }
  if (!early_weights && lane == 0)
    for (int i = 0; i < npre; ++i) issue(i);
  if (x_bulk) {
    if (!mbar_wait_bounded(xbar, 0, g.err)) abort_flag = 1;
  } else {
    for (int k = threadIdx.x; k < g.xbytes / 2; k += blockDim.x)
      reinterpret_cast<uint16_t*>(xraw)[k] = reinterpret_cast<const uint16_t*>(x)[k];
    __syncthreads();
  }
  prepare_x<D, XB>(xraw, g.nb, xrec, warp, nwarps, lane);
  __syncthreads();

  for (int i = 0; i < my_tiles; ++i) {
    const int st = i % g.stages;
    const int t = first + i * tile_stride;
    if (!abort_flag && !mbar_wait_bounded(&full[st], uint32_t(i / g.stages) & 1u, g.err)) abort_flag = 1;
    __syncwarp();
    const uint8_t* buf = ring + size_t(st) * g.stage_bytes;
    const uint32_t row_off = uint32_t(r * g.row_bytes);
    float yacc = 0.f;
    for (int b = v; b < g.nb; b += 4) {
      const uint32_t* rec = xrec + b * RW;
      int aA[2][D], aB[2][D];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) aA[h][d] = aB[h][d] = 0;
      // block start inside the buffer, and its offset from a 4-byte boundary (0 or 2)
      const uint32_t boff = row_off + 66u * uint32_t(b);
      const uint32_t fs = (boff & 3u) * 8u;
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(buf + (boff & ~3u));
      uint32_t nxt = aw[0];
#pragma unroll 4
      for (int wi = 0; wi < 16; ++wi) {
        const uint32_t cur = nxt;
        nxt = aw[wi + 1];
        const uint32_t w = __funnelshift_r(cur, nxt, fs) ^ 0x55555555u;
        uint32_t xw[4 * D];
#pragma unroll
        for (int k = 0; k < D; ++k) {
          const uint4 q = *reinterpret_cast<const uint4*>(rec + (wi * 4) * D + 4 * k);
          xw[4 * k] = q.x; xw[4 * k + 1] = q.y; xw[4 * k + 2] = q.z; xw[4 * k + 3] = q.w;
        }
        const uint32_t w2 = w >> 2;
        const uint32_t m0 = w & 0x03030303u, m1 = w2 & 0x03030303u;
        const uint32_t m2 = w & 0x30303030u, m3 = w2 & 0x30303030u;
        const int h = wi & 1;
#pragma unroll
        for (int d = 0; d < D - 1; ++d) {
          aA[h][d] = dp4a_uu(m0, xw[0 * D + d], aA[h][d]);
          aA[h][d] = dp4a_uu(m1, xw[1 * D + d], aA[h][d]);
          aB[h][d] = dp4a_uu(m2, xw[2 * D + d], aB[h][d]);
          aB[h][d] = dp4a_uu(m3, xw[3 * D + d], aB[h][d]);
        }
        aA[h][D - 1] = dp4a_us(m0, xw[0 * D + D - 1], aA[h][D - 1]);
        aA[h][D - 1] = dp4a_us(m1, xw[1 * D + D - 1], aA[h][D - 1]);
        aB[h][D - 1] = dp4a_us(m2, xw[2 * D + D - 1], aB[h][D - 1]);
        aB[h][D - 1] = dp4a_us(m3, xw[3 * D + D - 1], aB[h][D - 1]);
      }
      const int* sums = reinterpret_cast<const int*>(rec + 64 * D);
      float p = 0.f, sc = 1.f;
#pragma unroll
      for (int d = 0; d < D; ++d) {
        p += float(sums[d] - (aA[0][d] + aA[1][d] + ((aB[0][d] + aB[1][d]) >> 4))) * sc;
        sc *= 256.f;
      }
      const float* f = reinterpret_cast<const float*>(rec + 64 * D + D);
      const float dsc = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(buf + boff + 64)));
      yacc += dsc * ((p * f[0]) * f[1]);
    }
    // the four lanes of a row hold blocks b = v (mod 4); add them (same order on all four)
    yacc += __shfl_xor_sync(0xffffffffu, yacc, 8);
    yacc += __shfl_xor_sync(0xffffffffu, yacc, 16);
    __syncwarp();
    if (lane == 0 && i + g.stages < my_tiles) issue(i + g.stages);
    const int row = t * kRows + r;
    if (v == 0 && row < g.N) y[row] = yacc;
  }
  if (abort_flag && lane == 0) {
    for (int j = 0; j < my_tiles && j < g.stages; ++j) mbar_wait_bounded(&full[j], 0, nullptr);
    if (warp == 0) mbar_wait_bounded(xbar, 0, nullptr);
  }
}

template <int D>
bool plan(Geom& g, int64_t N, int64_t K, int esize, int max_smem, int nsm) {
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.N = int(N);
  g.K = int(K);
  g.nb = int(K / 256);
  g.row_bytes = int64_t(g.nb) * 66;
  g.xbytes = int(K * esize);
  g.ntiles = int((N + kRows - 1) / kRows);
  // + 4 bytes so the funnel-shift read of the last word stays inside the buffer
  g.stage_bytes = uint32_t(up(uint64_t(kRows) * g.row_bytes + 4, 128));
  // one CTA per SM with an even share of the tiles; as many warps as tiles
  // (at most 16), then the deepest ring that fits
  const int64_t grid = std::min<int64_t>(g.ntiles, nsm);
  const int64_t per_cta = (g.ntiles + grid - 1) / grid;
  for (int wpb = int(std::min<int64_t>(16, per_cta)); wpb >= 1; --wpb) {
    g.wpb = wpb;
    const uint64_t lim = uint64_t(max_smem);
    const int64_t tiles_per_warp = (per_cta + wpb - 1) / wpb;
    for (int st = int(std::min<int64_t>(3, std::max<int64_t>(1, tiles_per_warp))); st >= 1; --st) {
      uint64_t off = 0;
      g.off_bar = uint32_t(off);
      off = up(off + 8ull * (wpb * st + 1), 128);
      g.off_stage = uint32_t(off);
      off = up(off + uint64_t(wpb) * st * g.stage_bytes, 128);
      g.off_rec = uint32_t(off);
      off = up(off + 4ull * g.nb * Rec<D>::kWords, 128);
      g.off_xraw = uint32_t(off);
      off = up(off + uint64_t(g.xbytes), 128);
      if (off <= lim) {
        g.stages = st;
        g.smem = uint32_t(off);
        return true;
      }
    }
  }
  return false;
}

struct Plan {
  Geom g;
  int grid, threads;
};

template <int D, bool XB>
cudaError_t run(const uint8_t* packed, const void* x, float* y, int64_t N, int64_t K, cudaStream_t st) {
  auto kern = gemv_tq2_0_kernel<D, XB>;
  static PlanCache<Plan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  Plan p{};
  if (!cache.get(dev, N, K, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int nsm = sm_count();
    if (!plan<D>(p.g, N, K, XB ? 2 : 4, max_optin - 1024, nsm)) return cudaErrorInvalidConfiguration;
    cudaError_t e = raise_smem_cap(kern, dev, max_optin - 1024);
    if (e != cudaSuccess) return e;
    p.threads = 32 * p.g.wpb;
    p.grid = int(std::min<int64_t>(p.g.ntiles, nsm));
    p.g.err = dev_error_ptr();
    cache.put(dev, N, K, p);
  }
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(p.grid), dim3(p.threads), p.g.smem, st, pdl, packed, x, y, p.g, pdl ? 1 : 0);
}

}  // namespace

cudaError_t launch_gemv_tq2_0(const uint8_t* packed, const void* x, bl_dtype xt, float* y, int64_t N, int64_t K,
                              cudaStream_t s) {
  if (xt == BL_BF16) return run<3, true>(packed, x, y, N, K, s);
  return run<4, false>(packed, x, y, N, K, s);
}

}  // namespace bl
