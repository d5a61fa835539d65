// i2_s GEMV, one token: y[n] = scale * sum_k w[n,k] x[k]
// ("Hesper/Layers/BitLinear", sections "i2_s Packing Format" and
// "BitLinear Mathematics").
//
// Work decomposition.  A warp owns a tile of 16 rows: lanes l and l+16 both
// work on row l of the tile and take alternate 128-element groups of the
// warp's group range; their sums are added with one shuffle.  When rows are
// few the group range of a tile is split over `wk` warps of the CTA and
// their row sums are added in warp order.  Each row's slice is bulk-copied
// (cp.async.bulk) into a shared-memory row whose stride is an odd number of
// 16-byte units, so the 128-bit reads of every 8-lane phase hit distinct
// banks.  The activation digits of a group are read by broadcast (at most
// two addresses per instruction).  Row tiles of a warp stream through a ring
// of `stages` buffers completed by mbarriers (bounded waits).  The
// activation vector itself arrives by one bulk copy issued right after the
// wait on the previous kernel.
//
// Decode.  A 32-bit word of a group holds bytes p..p+3; bits (7-2t):(6-2t)
// of byte p are the code of element 32t+p.  Byte masks of the codes:
//   shift 0 (elements 96+p): w & 0x03030303         -> code
//   shift 2 (elements 64+p): (w >> 2) & 0x03030303  -> code
//   shift 4 (elements 32+p): w & 0x30303030         -> 16*code
//   shift 6 (elements p)   : (w >> 2) & 0x30303030  -> 16*code
// go to dp4a against the activation digits of those elements.  Codes are
// c = w + 1, so sum_k w_k X_k = sum_k c_k X_k - sum_k X_k.
//
// Activations.  Once per CTA, x is turned into exact fixed-point integers
// X = rint(x * 2^F_g) with one exponent per 128-element group g chosen from
// the group's max|x| so that |X| < 2^(8D-1), and stored as the D bytes of X
// in two's complement (X = sum_{d<D-1} u_d 256^d + s_{D-1} 256^(D-1) with
// unsigned low bytes u_d and a signed top byte).  D = 4 for fp32 input
// (fp32 values within 7 binades of the group maximum are carried exactly,
// smaller ones with absolute error <= 2^-32 * 2^ceil(log2 max)), D = 3 for
// bf16 input (exact within 15 binades).  Products and sums over a group are
// exact integers; each group sum is converted to fp32 once, scaled by
// 2^-F_g and added.
#include <algorithm>

#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kRows = 16;  // rows per warp tile (two lanes per row)

struct Geom {
  int N, K, nC;        // rows, columns, 128-element groups per row
  int wk, wr;          // warps per row tile (K split), row tiles per CTA
  int stages;          // ring depth per warp
  int ntiles;          // ceil(N / kRows)
  int rowstride;       // bytes per row in a ring buffer (odd multiple of 16)
  int xbytes;          // bytes of x (K * element size)
  uint32_t stage_bytes;
  uint32_t off_bar, off_stage, off_part, off_x, off_xraw, smem;
  unsigned int* err;
};

// Per-group activation record: [8 words][4 shifts][D digits] u32, then D
// digit sums (int) and two fp32 factors whose product is 2^-F_g.
template <int D>
struct Rec {
  static constexpr int kWords = (32 * D + D + 2 + 3) / 4 * 4;  // u32 per record, 16-byte multiple
};

template <int D, bool XB>
__device__ __forceinline__ void prepare_x(const void* xv, int nC, uint32_t* xrec, int warp, int nwarps, int lane) {
  constexpr int RW = Rec<D>::kWords;
  for (int c = warp; c < nC; c += nwarps) {
    // lane l holds elements 4l..4l+3 of group c: shift class t = l/8
    // (elements 32t..32t+31), bytes 4w..4w+3 with w = l%8.  xv is 8-byte
    // (bf16) or 16-byte (fp32) aligned here.
    float v[4];
    const int e0 = c * 128 + 4 * lane;
    if (XB) {
      const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(xv) + e0);
      v[0] = __uint_as_float(u.x << 16);
      v[1] = __uint_as_float(u.x & 0xFFFF0000u);
      v[2] = __uint_as_float(u.y << 16);
      v[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
      const float4 u = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xv) + e0);
      v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    // non-negative floats order like their bit patterns
    const float m = __uint_as_float(redux_max_u32(
        __float_as_uint(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))))));
    const int F = m > 0.f ? (8 * D - 1) - exponent_of(m) : 0;
    // x * 2^F as two exact power-of-two multiplies (each factor a normal float)
    const int fa = F / 2, fb = F - fa;
    const float sA = exp2i(fa), sB = exp2i(fb);
    int X[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      constexpr int kLim = int((1u << (8 * D - 1)) - 1u);  // keep the top byte signed
      X[b] = max(-kLim, min(kLim, __float2int_rn(__fmul_rn(__fmul_rn(v[b], sA), sB))));
    }
    uint32_t* rec = xrec + c * RW;
    const int t = lane >> 3, w = lane & 7, sh = 3 - t;
#pragma unroll
    for (int d = 0; d < D; ++d) {
      // byte d of the four values, element b in byte b
      const uint32_t sel = uint32_t(d) | (uint32_t(d + 4) << 4);
      const uint32_t lo = __byte_perm(uint32_t(X[0]), uint32_t(X[1]), sel);
      const uint32_t hi = __byte_perm(uint32_t(X[2]), uint32_t(X[3]), sel);
      const uint32_t dig = __byte_perm(lo, hi, 0x5410);
      rec[(w * 4 + sh) * D + d] = dig;
      const int s = redux_add(d == D - 1 ? dp4a_us(0x01010101u, dig, 0) : dp4a_uu(0x01010101u, dig, 0));
      if (lane == 0) reinterpret_cast<int*>(rec)[32 * D + d] = s;
    }
    if (lane == 0) {
      reinterpret_cast<float*>(rec)[32 * D + D] = exp2i(-fa);
      reinterpret_cast<float*>(rec)[32 * D + D + 1] = exp2i(-fb);
    }
  }
}

template <int D, bool XB, bool YB>
__global__ void __launch_bounds__(512) gemv_i2s_kernel(const uint8_t* __restrict__ packed, const void* __restrict__ x,
                                                       void* __restrict__ y, Geom g, int early_weights) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RW = Rec<D>::kWords;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int rt = warp / g.wk;  // row tile slot of this warp
  const int ks = warp % g.wk;  // group range of this warp
  const int c0 = ks * g.nC / g.wk, c1 = (ks + 1) * g.nC / g.wk;
  const int nchunks = c1 - c0;
  const int r = lane & (kRows - 1);  // row of the tile
  const int u = lane >> 4;            // which alternate groups
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar) + warp * g.stages;
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + g.off_bar) + nwarps * g.stages;
  uint64_t* tbar = xbar + 1 + rt;  // row-tile slot barrier: the wk warps of a tile meet here
  uint8_t* ring = smem + g.off_stage + size_t(warp) * g.stages * g.stage_bytes;
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  uint32_t* xrec = reinterpret_cast<uint32_t*>(smem + g.off_x);
  uint8_t* xraw = smem + g.off_xraw;
  __shared__ int abort_flag;

  const int tile_stride = int(gridDim.x) * g.wr;
  const int first = int(blockIdx.x) * g.wr + rt;
  const int my_tiles = first < g.ntiles ? (g.ntiles - 1 - first) / tile_stride + 1 : 0;
  const uint32_t slice_bytes = uint32_t(nchunks) * 32;
  const int64_t row_bytes = g.K / 4;

  // lanes 0..15 copy their row's group range of local tile i into ring buffer i % stages
  auto issue = [&](int i) {
    const int t = first + i * tile_stride;
    const int s = i % g.stages;
    const int row = t * kRows + r;
    const int nrows = min(kRows, g.N - t * kRows);
    if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(nrows) * slice_bytes);
    __syncwarp();
    if (u == 0 && row < g.N)
      bulk_g2s(ring + size_t(s) * g.stage_bytes + size_t(r) * g.rowstride, packed + int64_t(row) * row_bytes + 32 * c0,
               slice_bytes, &full[s], policy_evict_first());
  };

  if (lane == 0)
    for (int s = 0; s < g.stages; ++s) mbar_init(&full[s], 1);
  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    for (int k = 0; k < g.wr; ++k) mbar_init(xbar + 1 + k, 32 * g.wk);
    abort_flag = 0;
  }
  fence_barrier_init();
  __syncthreads();
  const int npre = min(my_tiles, g.stages);
  if (early_weights)
    for (int i = 0; i < npre; ++i) issue(i);
  pdl_wait();
  // activations: one bulk copy when aligned, else plain loads into the same buffer
  const bool x_bulk = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  if (threadIdx.x == 0 && x_bulk) {
    mbar_arrive_expect_tx(xbar, uint32_t(g.xbytes));
    bulk_g2s(xraw, x, uint32_t(g.xbytes), xbar, policy_evict_first());
  }
  if (!early_weights)
    for (int i = 0; i < npre; ++i) issue(i);
  if (x_bulk) {
    if (!mbar_wait_bounded(xbar, 0, g.err)) abort_flag = 1;
  } else {
    for (int k = threadIdx.x; k < g.xbytes / 2; k += blockDim.x)
      reinterpret_cast<uint16_t*>(xraw)[k] = reinterpret_cast<const uint16_t*>(x)[k];
    __syncthreads();
  }
  prepare_x<D, XB>(xraw, g.nC, xrec, warp, nwarps, lane);
  const float wscale = *reinterpret_cast<const float*>(packed + int64_t(g.N) * row_bytes);
  __syncthreads();
  pdl_launch_dependents();

  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % g.stages;
    const int t = first + i * tile_stride;
    if (!abort_flag && !mbar_wait_bounded(&full[s], uint32_t(i / g.stages) & 1u, g.err)) abort_flag = 1;
    __syncwarp();
    const uint8_t* myrow = ring + size_t(s) * g.stage_bytes + size_t(r) * g.rowstride;
    float yacc = 0.f;
    for (int cc = u; cc < nchunks; cc += 2) {
      const uint32_t* rec = xrec + (c0 + cc) * RW;
      // two independent accumulator sets (one per 16-byte half) shorten the dp4a chains
      int aA[2][D], aB[2][D];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int d = 0; d < D; ++d) aA[h][d] = aB[h][d] = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 wv = *reinterpret_cast<const uint4*>(myrow + 32 * cc + 16 * h);
        const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // digits of word 4h+j: [4 shifts][D] u32, shared by the lanes on this group
          uint32_t xw[4 * D];
#pragma unroll
          for (int k = 0; k < D; ++k) {
            const uint4 q = *reinterpret_cast<const uint4*>(rec + ((4 * h + j) * 4) * D + 4 * k);
            xw[4 * k] = q.x; xw[4 * k + 1] = q.y; xw[4 * k + 2] = q.z; xw[4 * k + 3] = q.w;
          }
          const uint32_t w = wds[j], w2 = w >> 2;
          const uint32_t m0 = w & 0x03030303u, m1 = w2 & 0x03030303u;
          const uint32_t m2 = w & 0x30303030u, m3 = w2 & 0x30303030u;
#pragma unroll
          for (int d = 0; d < D - 1; ++d) {  // unsigned low bytes
            aA[h][d] = dp4a_uu(m0, xw[0 * D + d], aA[h][d]);
            aA[h][d] = dp4a_uu(m1, xw[1 * D + d], aA[h][d]);
            aB[h][d] = dp4a_uu(m2, xw[2 * D + d], aB[h][d]);
            aB[h][d] = dp4a_uu(m3, xw[3 * D + d], aB[h][d]);
          }
          aA[h][D - 1] = dp4a_us(m0, xw[0 * D + D - 1], aA[h][D - 1]);  // signed top byte
          aA[h][D - 1] = dp4a_us(m1, xw[1 * D + D - 1], aA[h][D - 1]);
          aB[h][D - 1] = dp4a_us(m2, xw[2 * D + D - 1], aB[h][D - 1]);
          aB[h][D - 1] = dp4a_us(m3, xw[3 * D + D - 1], aB[h][D - 1]);
        }
      }
      const int* sums = reinterpret_cast<const int*>(rec + 32 * D);
      float p = 0.f, sc = 1.f;
#pragma unroll
      for (int d = 0; d < D; ++d) {
        p += float(aA[0][d] + aA[1][d] + ((aB[0][d] + aB[1][d]) >> 4) - sums[d]) * sc;
        sc *= 256.f;
      }
      const float* f = reinterpret_cast<const float*>(rec + 32 * D + D);
      yacc += (p * f[0]) * f[1];
    }
    // lanes l and l+16 hold the two halves of row l (same order on both)
    yacc += __shfl_xor_sync(0xffffffffu, yacc, 16);
    __syncwarp();
    if (i + g.stages < my_tiles) issue(i + g.stages);
    const int row = t * kRows + r;
    if (g.wk == 1) {
      if (u == 0 && row < g.N) {
        const float yv = yacc * wscale;
        if (YB)
          reinterpret_cast<uint16_t*>(y)[row] = f32_to_bf16_bits_rn(yv);
        else
          reinterpret_cast<float*>(y)[row] = yv;
      }
    } else {
      float* pp = part + ((rt * 2 + (i & 1)) * g.wk) * kRows;
      if (u == 0) pp[ks * kRows + r] = yacc;
      // all wk warps of the tile arrive and wait, so none can run a tile ahead
      mbar_arrive(tbar);
      if (!mbar_wait_bounded(tbar, uint32_t(i) & 1u, g.err)) abort_flag = 1;
      if (ks == 0 && u == 0 && row < g.N) {
        float acc = 0.f;
        for (int k = 0; k < g.wk; ++k) acc += pp[k * kRows + r];
        const float yv = acc * wscale;
        if (YB)
          reinterpret_cast<uint16_t*>(y)[row] = f32_to_bf16_bits_rn(yv);
        else
          reinterpret_cast<float*>(y)[row] = yv;
      }
    }
  }
  if (abort_flag && lane == 0) {
    // let copies still in flight land (bounded) before the CTA exits
    for (int j = 0; j < my_tiles && j < g.stages; ++j) mbar_wait_bounded(&full[j], 0, nullptr);
    if (warp == 0) mbar_wait_bounded(xbar, 0, nullptr);
  }
}

template <int D>
bool plan(Geom& g, int64_t N, int64_t K, int esize, int max_smem, int nsm) {
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.N = int(N);
  g.K = int(K);
  g.nC = int(K / 128);
  g.xbytes = int(K * esize);
  g.ntiles = int((N + kRows - 1) / kRows);
  // Split the groups of a tile over up to 16 warps while every warp keeps
  // at least two groups and there are fewer than ~16 warps per SM; then put
  // as many row tiles in a CTA as keep it at <= 16 warps without dropping
  // below one CTA per SM.  More warps per CTA also spread the per-CTA
  // activation preparation thinner.
  int wk = 1;
  while (wk < 16 && int64_t(g.ntiles) * wk < 16LL * nsm && g.nC / (wk + 1) >= 2) ++wk;
  g.wk = wk;
  int wr = std::max(1, 16 / wk);
  while (wr > 1 && (g.ntiles + wr - 1) / wr < nsm) --wr;
  g.wr = wr;
  const int max_chunks = (g.nC + wk - 1) / wk;
  int rs = int(up(uint64_t(max_chunks) * 32, 16));
  if (((rs / 16) & 1) == 0) rs += 16;
  g.rowstride = rs;
  g.stage_bytes = uint32_t(up(uint64_t(kRows) * rs, 128));
  const int warps = g.wk * g.wr;
  const int64_t tiles_per_warp = (g.ntiles + int64_t(g.wr) * nsm - 1) / (int64_t(g.wr) * nsm);
  for (int st = int(std::min<int64_t>(3, std::max<int64_t>(1, tiles_per_warp))); st >= 1; --st) {
    uint64_t off = 0;
    g.off_bar = uint32_t(off);
    off = up(off + 8ull * (warps * st + 1 + g.wr), 128);
    g.off_stage = uint32_t(off);
    off = up(off + uint64_t(warps) * st * g.stage_bytes, 128);
    g.off_part = uint32_t(off);
    off = up(off + (g.wk > 1 ? 4ull * g.wr * 2 * g.wk * kRows : 0), 128);
    g.off_x = uint32_t(off);
    off = up(off + 4ull * g.nC * Rec<D>::kWords, 128);
    g.off_xraw = uint32_t(off);
    off = up(off + uint64_t(g.xbytes), 128);
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
  bool ok;
};

template <int D, bool XB, bool YB>
cudaError_t run(const uint8_t* packed, const void* x, void* y, int64_t N, int64_t K, cudaStream_t st) {
  auto kern = gemv_i2s_kernel<D, XB, YB>;
  static PlanCache<Plan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  Plan p;
  if (!cache.get(dev, N, K, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int nsm = sm_count();
    p.ok = plan<D>(p.g, N, K, XB ? 2 : 4, max_optin - 1024, nsm);
    if (!p.ok) return cudaErrorInvalidConfiguration;
    // the cap is a property of the kernel, shared by every shape: raise it to the maximum once
    cudaError_t e = raise_smem_cap(kern, dev, max_optin - 1024);
    if (e != cudaSuccess) return e;
    p.threads = 32 * p.g.wk * p.g.wr;
    int blocks_per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kern, p.threads, p.g.smem);
    if (blocks_per_sm < 1) blocks_per_sm = 1;
    p.grid = (p.g.ntiles + p.g.wr - 1) / p.g.wr;
    if (p.grid > nsm * blocks_per_sm) p.grid = nsm * blocks_per_sm;
    p.g.err = dev_error_ptr();
    cache.put(dev, N, K, p);
  }
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(p.grid), dim3(p.threads), p.g.smem, st, pdl, packed, x, y, p.g, pdl ? 1 : 0);
}

}  // namespace

cudaError_t launch_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                            int64_t K, cudaStream_t s) {
  const bool xb = xt == BL_BF16, yb = yt == BL_BF16;
  if (xb) return yb ? run<3, true, true>(packed, x, y, N, K, s) : run<3, true, false>(packed, x, y, N, K, s);
  return yb ? run<4, false, true>(packed, x, y, N, K, s) : run<4, false, false>(packed, x, y, N, K, s);
}

}  // namespace bl
