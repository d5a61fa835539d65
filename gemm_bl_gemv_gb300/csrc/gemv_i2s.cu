// i2_s GEMV, one token: y[n] = scale * sum_k w[n,k] x[k]
// ("Hesper/Layers/BitLinear", sections "i2_s Packing Format" and
// "BitLinear Mathematics").
//
// Work decomposition.  The grid has one CTA per SM (fewer when N is small)
// and CTA c takes an equal contiguous range of rows (N/grid, rounded up for
// the first N % grid CTAs), so no SM holds more than one row above its
// share.  A CTA covers its rows with tiles of 16 (the last may be partial);
// when only a few rows (<= kExtraMax) are left over they are taken one row
// at a time instead, which costs about 1/16 of a tile per row.  The unit of
// work is one 128-element group of a tile (or of a single row); the tile
// units of the CTA are split evenly over its 16 warps, and so are the
// single-row units.  In a tile, lanes l and l+16 both work on row l and
// take alternate groups; their sums meet with one shuffle.  For a single
// row, lane (w, t) takes word w of each group and the codes of shift class
// t (its integer sum over its 4 elements is exact), and the warp adds its
// lanes at the end.  A tile or row cut between
// warps is summed in warp order in shared memory.  Nothing leaves the CTA
// before it is final, so results do not depend on timing.
//
// Staging.  A warp's units stream through a ring of `stages` buffers, one
// chunk (up to S groups of one tile or row) per buffer: each row's bytes
// arrive by a bulk copy (cp.async.bulk) into a shared-memory row whose
// stride is an odd number of 16-byte units, so the 128-bit reads of an
// 8-lane phase hit distinct banks; buffers complete on mbarriers (bounded
// waits).  With programmatic dependent launch the first chunks are
// requested before the wait on the previous kernel, since the weights do
// not depend on it.
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
// bf16 input with fp32 output (exact within 15 binades) and D = 2 for bf16
// input and output (exact within 7 binades, error <= 2^-16 * 2^ceil(log2
// max) below that: far under the output's own bf16 rounding, for a third
// fewer dp4a).  Products and sums over a group are
// exact integers; each group sum is converted to fp32 once, scaled by
// 2^-F_g and added.
#include <algorithm>

#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kRows = 16;     // rows per tile (two lanes per row)
constexpr int kWarps = 16;    // warps per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kExtraMax = 4;
constexpr int kResidentSmem = 110 * 1024;  // resident-mode budget: two CTAs fit on an SM  // leftover rows of a CTA taken one at a time (else a partial tile)

struct Geom {
  int N, K, nC;     // rows, columns, 128-element groups per row
  int grid;         // CTAs
  int q, rem;       // CTA c takes q rows, plus one when c < rem
  int resident;     // 1: the CTA's rows are copied whole, one bulk copy per row
  int S;            // groups per chunk at most (ring mode)
  int stages;       // ring depth per warp (ring mode)
  int tiles_max;    // tiles of a CTA at most
  int rows_alloc;   // rows of one matrix's resident block (tiles_max * 16 + kExtraMax)
  int rowstride;    // bytes per row in a shared-memory buffer (odd multiple of 16)
  uint32_t stage_bytes;
  uint32_t off_bar, off_stage, off_part, off_res, off_x, smem;
  unsigned int* err;
  // per call (single matrix only): residual added to y (y's dtype) and
  // RMSNorm weights (x's dtype) with epsilon; nullptr when not used
  const void* residual;
  const void* rms_w;
  float eps;
};

// Per-group activation record: [8 words][4 shifts][D digits] u32, then D
// digit sums (int) and two fp32 factors whose product is 2^-F_g.
template <int D>
struct Rec {
  static constexpr int kWords = (32 * D + D + 2 + 3) / 4 * 4;  // u32 per record, 16-byte multiple
};

// elements e0..e0+3 of x as fp32 (vec: x is 16-byte aligned)
template <bool XB>
__device__ __forceinline__ void load4(const void* x, bool vec, int e0, float (&v)[4]) {
  if (XB) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(x) + e0;
    uint32_t a, b;
    if (vec) {
      const uint2 q = *reinterpret_cast<const uint2*>(p);
      a = q.x;
      b = q.y;
    } else {
      a = uint32_t(p[0]) | (uint32_t(p[1]) << 16);
      b = uint32_t(p[2]) | (uint32_t(p[3]) << 16);
    }
    v[0] = __uint_as_float(a << 16);
    v[1] = __uint_as_float(a & 0xFFFF0000u);
    v[2] = __uint_as_float(b << 16);
    v[3] = __uint_as_float(b & 0xFFFF0000u);
  } else {
    const float* p = reinterpret_cast<const float*>(x) + e0;
    if (vec) {
      const float4 q = *reinterpret_cast<const float4*>(p);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      v[0] = p[0]; v[1] = p[1]; v[2] = p[2]; v[3] = p[3];
    }
  }
}

// One group's record from the 4 elements each lane holds: lane l holds
// elements 4l..4l+3, i.e. shift class t = l/8 (elements 32t..32t+31) and
// bytes 4w..4w+3 with w = l%8.  Whole warp.
template <int D>
__device__ __forceinline__ void prep_group(const float (&v)[4], uint32_t* rec, int lane) {
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

// Records of all nC groups, warp w taking groups w, w+16, ...; the loads of
// up to four groups are in flight together.
template <int D, bool XB>
__device__ __forceinline__ void prepare_x(const void* x, bool vec, int nC, uint32_t* xrec, int warp, int lane,
                                          const void* rmsw, bool wvec, float rinv) {
  constexpr int RW = Rec<D>::kWords;
  for (int c0 = warp; c0 < nC; c0 += 4 * kWarps) {
    float v[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (c0 + b * kWarps < nC) {
        load4<XB>(x, vec, (c0 + b * kWarps) * 128 + 4 * lane, v[b]);
        if (rmsw) {  // RMSNorm: x * rmsInv * weight
          float w[4];
          load4<XB>(rmsw, wvec, (c0 + b * kWarps) * 128 + 4 * lane, w);
#pragma unroll
          for (int i = 0; i < 4; ++i) v[b][i] = __fmul_rn(__fmul_rn(v[b][i], rinv), w[i]);
        }
      }
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (c0 + b * kWarps < nC) prep_group<D>(v[b], xrec + (c0 + b * kWarps) * RW, lane);
  }
}

// sum_k w_k x_k over one group of two rows: `wa`, `wb` hold the rows' 32
// packed bytes of the group, `rec` the group's activation record; the
// results are added to ya, yb.  Each digit word read from shared memory
// serves both rows.
template <int D>
__device__ __forceinline__ void group_dot2(const uint8_t* wa, const uint8_t* wb, const uint32_t* rec, float& ya,
                                           float& yb) {
  // [row][digit]: shift classes 0 and 1 (codes), 2 and 3 (16 * codes)
  int aA[2][D], aB[2][D];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int d = 0; d < D; ++d) aA[i][d] = aB[i][d] = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 va = *reinterpret_cast<const uint4*>(wa + 16 * h);
    const uint4 vb = *reinterpret_cast<const uint4*>(wb + 16 * h);
    const uint32_t wds[2][4] = {{va.x, va.y, va.z, va.w}, {vb.x, vb.y, vb.z, vb.w}};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // digits of word 4h+j: [4 shifts][D] u32, shared by the lanes on this group
      uint32_t xw[4 * D];
#pragma unroll
      for (int k = 0; k < D; ++k) {
        const uint4 q = *reinterpret_cast<const uint4*>(rec + ((4 * h + j) * 4) * D + 4 * k);
        xw[4 * k] = q.x; xw[4 * k + 1] = q.y; xw[4 * k + 2] = q.z; xw[4 * k + 3] = q.w;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t w = wds[i][j], w2 = w >> 2;
        const uint32_t m0 = w & 0x03030303u, m1 = w2 & 0x03030303u;
        const uint32_t m2 = w & 0x30303030u, m3 = w2 & 0x30303030u;
#pragma unroll
        for (int d = 0; d < D - 1; ++d) {  // unsigned low bytes
          aA[i][d] = dp4a_uu(m0, xw[0 * D + d], aA[i][d]);
          aA[i][d] = dp4a_uu(m1, xw[1 * D + d], aA[i][d]);
          aB[i][d] = dp4a_uu(m2, xw[2 * D + d], aB[i][d]);
          aB[i][d] = dp4a_uu(m3, xw[3 * D + d], aB[i][d]);
        }
        aA[i][D - 1] = dp4a_us(m0, xw[0 * D + D - 1], aA[i][D - 1]);  // signed top byte
        aA[i][D - 1] = dp4a_us(m1, xw[1 * D + D - 1], aA[i][D - 1]);
        aB[i][D - 1] = dp4a_us(m2, xw[2 * D + D - 1], aB[i][D - 1]);
        aB[i][D - 1] = dp4a_us(m3, xw[3 * D + D - 1], aB[i][D - 1]);
      }
    }
  }
  const int* sums = reinterpret_cast<const int*>(rec + 32 * D);
  const float* f = reinterpret_cast<const float*>(rec + 32 * D + D);
  float p[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float sc = 1.f;
    p[i] = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) {
      p[i] += float(aA[i][d] + (aB[i][d] >> 4) - sums[d]) * sc;  // aB is a multiple of 16
      sc *= 256.f;
    }
  }
  ya += (p[0] * f[0]) * f[1];
  yb += (p[1] * f[0]) * f[1];
}

template <bool YB>
__device__ __forceinline__ void store_y(void* y, int row, float v) {
  if (YB)
    reinterpret_cast<uint16_t*>(y)[row] = f32_to_bf16_bits_rn(v);
  else
    reinterpret_cast<float*>(y)[row] = v;
}

// Walks a warp's units: first its tile units [a0, a1), then its single-row
// units [b0, b1), in chunks of at most S groups that never cross a tile or
// row.  `idx` is the tile (phase 0) or single row (phase 1) of the chunk.
struct Cursor {
  int phase, at, end, idx, gg;
  int b0, b1, nC, S;
  __device__ __forceinline__ void start(int a0_, int a1_, int b0_, int b1_, int nC_, int S_) {
    b0 = b0_;
    b1 = b1_;
    nC = nC_;
    S = S_;
    phase = 0;
    set(a0_, a1_);
    if (at >= end) next_phase();
  }
  __device__ __forceinline__ void set(int a, int e) {
    at = a;
    end = e;
    idx = a / nC;
    gg = a - idx * nC;
  }
  __device__ __forceinline__ void next_phase() {
    if (phase == 0) {
      phase = 1;
      set(b0, b1);
      if (at < end) return;
    }
    phase = 2;
  }
  __device__ __forceinline__ bool done() const { return phase == 2; }
  __device__ __forceinline__ int len() const { return min(min(S, nC - gg), end - at); }
  __device__ __forceinline__ void advance(int n) {
    at += n;
    gg += n;
    if (gg == nC) {
      gg = 0;
      ++idx;
    }
    if (at == end) next_phase();
  }
};

// NM = 1: y = scale * W x.  NM = 2: the fused gate/up product of the MLP,
// y = max(0, g)^2 * u with g = scale_g * W_g x and u = scale_u * W_u x
// ("Hesper/Layers/BitLinear", "Fused Gate+Up+ReLU²×Mul M=1 Kernel"): both
// matrices' rows of the CTA's range are units of the same CTA, and the
// epilogue runs once both results of a row are final.
template <int D, bool XB, bool YB, int NM>
__global__ void __launch_bounds__(kThreads, 2) gemv_i2s_kernel(const uint8_t* __restrict__ packed,
                                                            const uint8_t* __restrict__ packed2,
                                                            const void* __restrict__ x, void* __restrict__ y, Geom g,
                                                            int early_weights) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RW = Rec<D>::kWords;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int ir = lane & (kRows - 1);  // row a lane < 16 copies into a ring buffer
  const int q = lane & 7;              // tile rows q and q+8 of this lane
  const int u = lane >> 3;             // groups u, u+4, ... of a chunk
  // ring mode: `stages` buffers per warp; resident mode: the CTA's rows, one
  // barrier per tile and one for the single rows
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar) + (g.resident ? 0 : warp * g.stages);
  uint8_t* ring = smem + g.off_stage + (g.resident ? size_t(0) : size_t(warp) * g.stages * g.stage_bytes);
  float* part_t = reinterpret_cast<float*>(smem + g.off_part);  // [kWarps][2][kRows]
  float* part_r = part_t + kWarps * 2 * kRows;                   // [kWarps][2]
  uint32_t* xrec = reinterpret_cast<uint32_t*>(smem + g.off_x);
  __shared__ int abort_flag;
  __shared__ int wspan[kWarps][4];  // first/last tile, first/last single row of each warp (-1: none)

  // rows of this CTA, covered by `ntile` tiles and `nextra` single rows
  const int c = blockIdx.x;
  const int r0 = c * g.q + min(c, g.rem);
  const int rows = g.q + (c < g.rem ? 1 : 0);
  int ntile = rows / kRows, nextra = rows % kRows;
  if (nextra > kExtraMax) {
    ++ntile;
    nextra = 0;
  }
  const int tile_rows = rows - nextra;
  // units run over NM matrices: virtual tile v is tile v % ntile of matrix
  // v / ntile, virtual single row likewise
  const int TU = NM * ntile * g.nC, RU = NM * nextra * g.nC;
  auto pk = [&](int m) { return (NM == 2 && m) ? packed2 : packed; };
  auto vsplit = [&](int v, int per, int& m) {
    m = (NM == 2 && v >= per) ? 1 : 0;
    return v - m * per;
  };
  const int nbar = ntile + 1;                           // resident barriers per matrix
  const size_t mat_bytes = size_t(g.rows_alloc) * g.rowstride;  // resident block per matrix
  auto split = [&](int n, int w) { return w * (n / kWarps) + min(w, n % kWarps); };
  const int ta = split(TU, warp), tb = split(TU, warp + 1);
  const int ra = split(RU, warp), rb = split(RU, warp + 1);
  const int64_t row_bytes = g.K / 4;

  Cursor ic;  // issue cursor, runs `stages` chunks ahead of the compute cursor (ring mode)
  ic.start(ta, tb, ra, rb, g.nC, g.S);
  if (g.resident) ic.phase = 2;
  int issued = 0;
  auto issue_next = [&]() {
    if (ic.done()) return;
    const int s = issued % g.stages;
    const int n = ic.len();
    uint8_t* dst = ring + size_t(s) * g.stage_bytes;
    int m;
    if (ic.phase == 0) {
      const int t = vsplit(ic.idx, ntile, m);
      const int nrows = min(kRows, tile_rows - t * kRows);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(nrows * n * 32));
      __syncwarp();
      if (lane < kRows && ir < nrows)
        bulk_g2s(dst + size_t(ir) * g.rowstride, pk(m) + int64_t(r0 + t * kRows + ir) * row_bytes + 32 * ic.gg,
                 uint32_t(n * 32), &full[s], policy_evict_first());
    } else if (lane == 0) {
      const int j = vsplit(ic.idx, nextra, m);
      mbar_arrive_expect_tx(&full[s], uint32_t(n * 32));
      bulk_g2s(dst, pk(m) + int64_t(r0 + tile_rows + j) * row_bytes + 32 * ic.gg, uint32_t(n * 32), &full[s],
               policy_evict_first());
    }
    ic.advance(n);
    ++issued;
  };

  if (g.resident) {
    if (int(threadIdx.x) < NM * nbar) mbar_init(&full[threadIdx.x], 1);
  } else if (lane == 0) {
    for (int s = 0; s < g.stages; ++s) mbar_init(&full[s], 1);
  }
  if (lane == 0) {
    wspan[warp][0] = tb > ta ? ta / g.nC : -1;
    wspan[warp][1] = tb > ta ? (tb - 1) / g.nC : -1;
    wspan[warp][2] = rb > ra ? ra / g.nC : -1;
    wspan[warp][3] = rb > ra ? (rb - 1) / g.nC : -1;
  }
  if (threadIdx.x == 0) abort_flag = 0;
  fence_barrier_init();
  __syncthreads();
  // resident mode: one bulk copy per row of the CTA, tile i completing on
  // barrier i and the single rows on barrier ntile
  auto issue_rows = [&]() {
    if (int(threadIdx.x) < NM * nbar) {
      const int b = int(threadIdx.x) % nbar;
      const int nr = b < ntile ? min(kRows, tile_rows - b * kRows) : nextra;
      mbar_arrive_expect_tx(&full[threadIdx.x], uint32_t(nr) * uint32_t(row_bytes));
    }
    if (int(threadIdx.x) < NM * rows) {
      const int m = int(threadIdx.x) / rows, t = int(threadIdx.x) % rows;
      bulk_g2s(ring + m * mat_bytes + size_t(t) * g.rowstride, pk(m) + int64_t(r0 + t) * row_bytes,
               uint32_t(row_bytes), &full[m * nbar + (t < tile_rows ? t / kRows : ntile)], policy_evict_first());
    }
  };
  if (early_weights) {
    if (g.resident)
      issue_rows();
    else
      for (int i = 0; i < g.stages; ++i) issue_next();
  }
  // let the next kernel's CTAs become resident now: they fetch their own
  // weights and then wait for this grid to complete before touching its outputs
  pdl_launch_dependents();
  pdl_wait();
  if (!early_weights) {
    if (g.resident)
      issue_rows();
    else
      for (int i = 0; i < g.stages; ++i) issue_next();
  }
  const bool xvec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  float rinv = 1.f;
  if (NM == 1 && g.rms_w) {
    // RMSNorm factor 1 / sqrt(mean(x^2) + eps): lanes, warps and the CTA sum
    // in a fixed order (every CTA gets the same value)
    __shared__ float ssq[kWarps];
    float part = 0.f;
    for (int c0 = warp; c0 < g.nC; c0 += kWarps) {
      float v[4];
      load4<XB>(x, xvec, c0 * 128 + 4 * lane, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) part = __fadd_rn(part, __fmul_rn(v[i], v[i]));
    }
    part = warp_sum(part);
    if (lane == 0) ssq[warp] = part;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot = __fadd_rn(tot, ssq[w]);
    rinv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, float(g.K)), g.eps)));
  }
  prepare_x<D, XB>(x, xvec, g.nC, xrec, warp, lane, NM == 1 ? g.rms_w : nullptr,
                   (reinterpret_cast<uintptr_t>(g.rms_w) & 15) == 0, rinv);
  const float wsc0 = *reinterpret_cast<const float*>(pk(0) + int64_t(g.N) * row_bytes);
  const float wsc1 = NM == 2 ? *reinterpret_cast<const float*>(pk(1) + int64_t(g.N) * row_bytes) : wsc0;
  float* res = reinterpret_cast<float*>(smem + g.off_res);  // NM == 2: [2][rows_alloc] scaled results
  // a row's final value: stored (NM == 1) or kept for the epilogue (NM == 2)
  auto emit = [&](int m, int row_local, float v) {
    if (NM == 1) {
      float out = v * wsc0;
      if (g.residual) {
        const int row = r0 + row_local;
        out += YB ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(g.residual)[row])
                  : reinterpret_cast<const float*>(g.residual)[row];
      }
      if (!abort_flag) store_y<YB>(y, r0 + row_local, out);
    } else {
      res[m * g.rows_alloc + row_local] = v * (m ? wsc1 : wsc0);
    }
  };
  __syncthreads();

  // ---- the warp's units, chunk by chunk -------------------------------------
  Cursor cc;
  cc.start(ta, tb, ra, rb, g.nC, g.resident ? g.nC : g.S);
  float yacc = 0.f, yacc2 = 0.f;  // tile rows q and q+8, or the single row
  const int lw = lane & 7, lsh = 3 - (lane >> 3);  // single rows: word and shift index of this lane
  for (int i = 0; !cc.done(); ++i) {
    const int s = i % g.stages;
    const int n = cc.len();
    const int phase = cc.phase, idx = cc.idx, gg = cc.gg;
    const int seg_lo = max(phase == 0 ? ta : ra, idx * g.nC);
    int m;
    const int loc = vsplit(idx, phase == 0 ? ntile : nextra, m);  // tile or single row within matrix m
    if (g.resident) {
      if (!abort_flag && !mbar_wait_bounded(&full[m * nbar + (phase == 0 ? loc : ntile)], 0, g.err)) abort_flag = 1;
    } else if (!abort_flag && !mbar_wait_bounded(&full[s], uint32_t(i / g.stages) & 1u, g.err)) {
      abort_flag = 1;
    }
    __syncwarp();
    // this chunk's bytes: group gg of the first row (+32 per group, + rowstride per row)
    const uint8_t* buf = g.resident
                             ? ring + m * mat_bytes + size_t(phase == 0 ? loc * kRows : tile_rows + loc) * g.rowstride + 32 * gg
                             : ring + size_t(s) * g.stage_bytes;
    if (phase == 0) {
      const uint8_t* rowa = buf + size_t(q) * g.rowstride;
      const uint8_t* rowb = rowa + size_t(8) * g.rowstride;
      for (int k = u; k < n; k += 4) group_dot2<D>(rowa + 32 * k, rowb + 32 * k, xrec + (gg + k) * RW, yacc, yacc2);
    } else {
      for (int k = 0; k < n; ++k) {
        const uint32_t* rec = xrec + (gg + k) * RW;
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(buf + 32 * k + 4 * lw);
        const uint32_t m = (wd >> (2 * lsh)) & 0x03030303u;
        // sum over this lane's 4 elements of (code - 1) * X, exact per digit;
        // a zero-weight row gives exactly zero in every lane
        float p = 0.f, sc = 1.f;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          const uint32_t dig = rec[(lw * 4 + lsh) * D + d];
          const int a = d == D - 1 ? dp4a_us(m, dig, 0) - dp4a_us(0x01010101u, dig, 0)
                                   : dp4a_uu(m, dig, 0) - dp4a_uu(0x01010101u, dig, 0);
          p += float(a) * sc;
          sc *= 256.f;
        }
        const float* f = reinterpret_cast<const float*>(rec + 32 * D + D);
        yacc += (p * f[0]) * f[1];
      }
    }
    __syncwarp();
    if (!g.resident) issue_next();  // the buffer just read takes chunk i + stages
    cc.advance(n);
    const bool seg_end = gg + n == g.nC || cc.phase != phase;
    if (!seg_end) continue;
    const bool whole = seg_lo == idx * g.nC && gg + n == g.nC;
    const int kind = seg_lo == (phase == 0 ? ta : ra) ? 0 : 1;
    if (phase == 0) {
      // the four group classes of rows q and q+8: lanes q, q+8, q+16, q+24
      float va = yacc + __shfl_xor_sync(0xffffffffu, yacc, 8);
      float vb = yacc2 + __shfl_xor_sync(0xffffffffu, yacc2, 8);
      va += __shfl_xor_sync(0xffffffffu, va, 16);
      vb += __shfl_xor_sync(0xffffffffu, vb, 16);
      const int nrows = min(kRows, tile_rows - loc * kRows);
      if (u == 0) {
        if (whole) {
          if (q < nrows) emit(m, loc * kRows + q, va);
          if (q + 8 < nrows) emit(m, loc * kRows + q + 8, vb);
        } else {
          part_t[(warp * 2 + kind) * kRows + q] = va;
          part_t[(warp * 2 + kind) * kRows + q + 8] = vb;
        }
      }
    } else {
      const float v = warp_sum(yacc);
      if (lane == 0) {
        if (whole) {
          emit(m, tile_rows + loc, v);
        } else {
          part_r[warp * 2 + kind] = v;
        }
      }
    }
    yacc = 0.f;
    yacc2 = 0.f;
  }
  __syncthreads();

  // ---- tiles and rows cut between warps: the first warp touching one sums
  //      the pieces in warp order.  Lane w (< 16) holds warp w's spans; a
  //      ballot gives the warps touching a tile, and the pieces of all 16
  //      warps are loaded at once (zero where a warp does not touch it: adding
  //      +0.0 in order changes no sum) ------------------------------------------
  int sp[4] = {-1, -1, -1, -1};
  if (lane < kWarps)
#pragma unroll
    for (int k = 0; k < 4; ++k) sp[k] = wspan[lane][k];
#pragma unroll
  for (int ph = 0; ph < 2; ++ph) {
    const int lo = ph == 0 ? ta : ra, hi = ph == 0 ? tb : rb;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = __shfl_sync(0xffffffffu, sp[2 * ph + k], warp);
      const int tf = __shfl_sync(0xffffffffu, sp[2 * ph], warp);
      if (hi <= lo || (k == 1 && t == tf)) continue;  // nothing, or one tile/row: stored as the first segment
      const int t0 = t * g.nC;
      if (lo <= t0 && t0 + g.nC <= hi) continue;  // whole inside this warp: already written
      const unsigned int touch = __ballot_sync(0xffffffffu, sp[2 * ph] >= 0 && sp[2 * ph] <= t && t <= sp[2 * ph + 1]);
      if ((__ffs(touch) - 1) != warp) continue;  // an earlier warp owns it
      float acc = 0.f;
      if (ph == 0) {
        if (lane < kRows) {
          float v[kWarps];
#pragma unroll
          for (int w2 = 0; w2 < kWarps; ++w2)
            v[w2] = (touch >> w2) & 1u ? part_t[(w2 * 2 + (w2 == warp ? k : 0)) * kRows + lane] : 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kWarps; ++w2) acc += v[w2];
        }
        int m;
        const int tl = vsplit(t, ntile, m);
        const int nrows = min(kRows, tile_rows - tl * kRows);
        if (lane < nrows) emit(m, tl * kRows + lane, acc);
      } else if (lane == 0) {
        float v[kWarps];
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) v[w2] = (touch >> w2) & 1u ? part_r[w2 * 2 + (w2 == warp ? k : 0)] : 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) acc += v[w2];
        int m;
        const int j = vsplit(t, nextra, m);
        emit(m, tile_rows + j, acc);
      }
    }
  }

  if (NM == 2) {
    // epilogue of the fused gate/up product: h = max(0, g)^2 * u
    __syncthreads();
    for (int i = threadIdx.x; i < rows; i += kThreads) {
      const float gv = fmaxf(res[i], 0.f), uv = res[g.rows_alloc + i];
      if (!abort_flag) store_y<YB>(y, r0 + i, (gv * gv) * uv);
    }
  }

  if (abort_flag && lane == 0) {
    // let copies still in flight land (bounded) before the CTA exits
    if (g.resident) {
      if (warp == 0)
        for (int j = 0; j < NM * nbar; ++j) mbar_wait_bounded(&full[j], 0, nullptr);
    } else {
      for (int j = 0; j < g.stages && j < issued; ++j) mbar_wait_bounded(&full[j], 0, nullptr);
    }
  }
}

template <int D, int NM>
bool plan(Geom& g, int64_t N, int64_t K, int max_smem, int nsm) {
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.N = int(N);
  g.K = int(K);
  g.nC = int(K / 128);
  g.grid = int(std::min<int64_t>(nsm, N));
  g.q = g.N / g.grid;
  g.rem = g.N % g.grid;
  // units per warp at most: the tiles of q+1 rows (or a partial tile) and a
  // few single rows, for each matrix
  const int rows = g.q + (g.rem ? 1 : 0);
  const int tiles = (rows + kRows - 1) / kRows;
  g.tiles_max = tiles;
  g.rows_alloc = tiles * kRows + kExtraMax;
  const long long per_warp =
      NM * (((long long)tiles * g.nC + kWarps - 1) / kWarps + (long long)kExtraMax * g.nC / kWarps + 1);
  const uint64_t fixed_x = up(4ull * g.nC * Rec<D>::kWords, 128);
  const uint64_t res_bytes = NM == 2 ? up(4ull * 2 * g.rows_alloc, 128) : 0;
  {
    // resident mode when the CTA's rows fit next to the activation records,
    // leaving room for a second CTA (the next kernel's) on the SM
    int rs = int(up(uint64_t(K / 4), 16));
    if (((rs / 16) & 1) == 0) rs += 16;
    uint64_t off = 0;
    const uint32_t off_bar = uint32_t(off);
    off = up(off + 8ull * NM * (tiles + 1), 128);
    const uint32_t off_stage = uint32_t(off);
    off = up(off + uint64_t(NM) * g.rows_alloc * rs, 128);
    const uint32_t off_part = uint32_t(off);
    off = up(off + 4ull * kWarps * 2 * (kRows + 1), 128);
    const uint32_t off_res = uint32_t(off);
    off += res_bytes;
    const uint32_t off_x = uint32_t(off);
    off += fixed_x;
    if (off <= uint64_t(std::min(max_smem, kResidentSmem)) && NM * g.rows_alloc <= kThreads) {
      g.resident = 1;
      g.S = g.nC;
      g.stages = 1;
      g.rowstride = rs;
      g.stage_bytes = 0;
      g.off_bar = off_bar;
      g.off_stage = off_stage;
      g.off_part = off_part;
      g.off_res = off_res;
      g.off_x = off_x;
      g.smem = uint32_t(off);
      return true;
    }
  }
  g.resident = 0;
  for (int S = int(std::min<long long>(8, std::max<long long>(1, per_warp))); S >= 1; S = S > 1 ? S / 2 : 0) {
    int rs = int(up(uint64_t(S) * 32, 16));
    if (((rs / 16) & 1) == 0) rs += 16;
    const uint32_t stage_bytes = uint32_t(up(uint64_t(kRows) * rs, 128));
    const long long chunks = (per_warp + S - 1) / S + 2 * NM;  // tile and phase boundaries add a few
    for (int st = int(std::min<long long>(3, std::max<long long>(1, chunks))); st >= 1; --st) {
      uint64_t off = 0;
      const uint32_t off_bar = uint32_t(off);
      off = up(off + 8ull * kWarps * st, 128);
      const uint32_t off_stage = uint32_t(off);
      off = up(off + uint64_t(kWarps) * st * stage_bytes, 128);
      const uint32_t off_part = uint32_t(off);
      off = up(off + 4ull * kWarps * 2 * (kRows + 1), 128);
      const uint32_t off_res = uint32_t(off);
      off += res_bytes;
      const uint32_t off_x = uint32_t(off);
      off += fixed_x;
      if (off <= uint64_t(max_smem)) {
        g.S = S;
        g.rowstride = rs;
        g.stage_bytes = stage_bytes;
        g.stages = st;
        g.off_bar = off_bar;
        g.off_stage = off_stage;
        g.off_part = off_part;
        g.off_res = off_res;
        g.off_x = off_x;
        g.smem = uint32_t(off);
        return true;
      }
    }
    if (S == 1) break;
  }
  return false;
}

struct Plan {
  Geom g;
  bool ok;
};

template <int D, bool XB, bool YB, int NM>
cudaError_t run(const uint8_t* packed, const uint8_t* packed2, const void* x, void* y, int64_t N, int64_t K,
                cudaStream_t st, const void* residual = nullptr, const void* rms_w = nullptr, float eps = 0.f) {
  auto kern = gemv_i2s_kernel<D, XB, YB, NM>;
  static PlanCache<Plan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  Plan p{};
  if (!cache.get(dev, N, K, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    p.ok = plan<D, NM>(p.g, N, K, max_optin - 1024, sm_count());
    if (!p.ok) return cudaErrorInvalidConfiguration;
    // the cap is a property of the kernel, shared by every shape: raise it to the maximum once
    cudaError_t e = raise_smem_cap(kern, dev, max_optin - 1024);
    if (e != cudaSuccess) return e;
    p.g.err = dev_error_ptr();
    cache.put(dev, N, K, p);
  }
  p.g.residual = residual;
  p.g.rms_w = rms_w;
  p.g.eps = eps;
  const bool pdl = overlap_enabled();
  return launch(kern, dim3(p.g.grid), dim3(kThreads), p.g.smem, st, pdl, packed, packed2, x, y, p.g, pdl ? 1 : 0);
}

}  // namespace

cudaError_t launch_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                            int64_t K, cudaStream_t s, const void* residual, const void* rms_w, float eps) {
  const cudaError_t e = launch_gemv_i2s_slot(packed, x, xt, y, yt, N, K, s, residual, rms_w, eps);
  if (e != cudaErrorNotSupported) return e;
  const bool xb = xt == BL_BF16, yb = yt == BL_BF16;
  if (xb)
    return yb ? run<2, true, true, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps)
              : run<3, true, false, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps);
  return yb ? run<4, false, true, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps)
            : run<4, false, false, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps);
}

cudaError_t launch_gemv_i2s_gate_up(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x, bl_dtype xt,
                                    void* h, bl_dtype ht, int64_t N, int64_t K, cudaStream_t s) {
  const cudaError_t e = launch_gemv_i2s_gate_up_slot(packed_gate, packed_up, x, xt, h, ht, N, K, s);
  if (e != cudaErrorNotSupported) return e;
  const bool xb = xt == BL_BF16, hb = ht == BL_BF16;
  if (xb)
    return hb ? run<2, true, true, 2>(packed_gate, packed_up, x, h, N, K, s)
              : run<3, true, false, 2>(packed_gate, packed_up, x, h, N, K, s);
  return hb ? run<4, false, true, 2>(packed_gate, packed_up, x, h, N, K, s)
            : run<4, false, false, 2>(packed_gate, packed_up, x, h, N, K, s);
}

}  // namespace bl
