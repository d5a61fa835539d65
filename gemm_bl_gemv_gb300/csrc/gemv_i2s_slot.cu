// i2_s GEMV, one token, activation-stationary form:
//   y[n] = scale * sum_k w[n,k] x[k]
// ("Hesper/Layers/BitLinear", sections "i2_s Packing Format" and "BitLinear
// Mathematics"); with two matrices, the fused gate/up product of the MLP
// ("Fused Gate+Up+ReLU²×Mul M=1 Kernel"): h = max(0, g)^2 * u.
//
// The grid has one CTA per SM (fewer when N is small); CTA c takes an equal
// contiguous range of rows (N / grid, one more for the first N % grid CTAs).
// Its rows (of both matrices for the fused product) arrive in shared memory
// by one bulk copy per row, issued before the wait on the previous kernel:
// the weights never depend on it.
//
// Activations.  After that wait, each 128-element group of x is turned, once
// per CTA, into exact fixed-point integers X = rint(x * 2^F_g) with
// 2^(8D-2) <= max|x_g| * 2^F_g < 2^(8D-1), stored as D byte digits (unsigned
// low digits, signed top digit).  D = 2 for bf16 x and bf16 y, 3 otherwise:
// bf16 values within 7 (D = 2) or 15 (D = 3) binades of the group maximum
// are exact; every other value (fp32 values with their 24-bit significands
// included) carries an absolute error of at most 2^-(8D-1) max|x_g|.  A warp converts two groups at a time (16 lanes, 8
// elements each) and writes the digits in the order the dot products read
// them.
//
// Slots.  A row's group is 32 bytes = 8 words; word j holds bytes 4j..4j+3,
// and bits (7-2t):(6-2t) of byte p are the code of element 32t + p.  A slot
// is W consecutive words of one group (W = 4 for D = 2, else 2: 16 W
// elements, 4 W D digit words).  Every thread owns one slot: it loads the
// slot's digits into registers once and then streams rows through them --
// for a row, one shared-memory load brings the slot's W code words, and per
// word four masks
//   w & 0x03030303          codes of elements 96 + p       (t = 3)
//   (w >> 2) & 0x03030303   codes of elements 64 + p       (t = 2)
//   w & 0x30303030          16 x codes of elements 32 + p  (t = 1)
//   (w >> 2) & 0x30303030   16 x codes of elements p       (t = 0)
// go to dp4a against the digits.  Codes are c = w + 1, so
// sum w X = sum c X - sum X, with the slot's digit sums stored beside its
// digits.  The slot sum is an exact integer; it is scaled by 2^-F_g (exact)
// and written to shared memory as the row's partial.  The threads sharing a
// slot take every nl-th row (nl = threads per slot), so every thread does
// the same work to within one row.  Finally one warp per output adds a
// row's partials in slot order (lanes in fixed strides, then a fixed
// butterfly), so results do not depend on timing.  For the fused gate/up,
// when a whole warp holds no slot, the gate and up rows of the first half of
// the outputs are computed first and that warp sums those outputs (a lane
// per output, slots in order) while the other warps compute the rest.
#include <algorithm>

#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCoResident = 110 * 1024;  // two CTAs (this launch and the next) fit on an SM

template <int D>
struct Slot {
  static constexpr int W = D == 2 ? 4 : 2;      // code words per slot
  static constexpr int kPerGroup = 8 / W;        // slots per 128-element group
  static constexpr int kDig = 4 * W * D;         // digit words per slot
  static constexpr int kTail = D + 2;            // D digit sums, two factors whose product is 2^-F
  // record stride: an odd number of 16-byte units, so that the 16-byte loads
  // of eight consecutive slots' records fall in distinct bank groups
  static constexpr int kUnits = ((kDig + kTail + 3) / 4) | 1;
  static constexpr int kStride = 4 * kUnits;     // u32 per slot record
};

struct SGeom {
  int N, K;           // rows, columns
  int ks;             // CTAs sharing a row range (a cluster), each taking 1/ks of K
  int nC, NS;         // 128-element groups and slots of a row in one CTA's share of K
  int grid, q, rem;   // cluster c takes q rows, plus one when c < rem
  int nl;             // threads per slot
  int RS;             // bytes per row in shared memory (this CTA's share: 32 nC)
  int PS;             // partials per row in shared memory (NS rounded up to odd: conflict-free row reads)
  int tpr;            // threads adding one row's partials (a power of two <= 32 / NM)
  int ovl;            // NM == 2 and a whole warp holds no slot: the last warp sums half of the outputs early
  uint32_t off_rec, off_part, off_sum, smem;
  unsigned int* err;
  unsigned long long wait_ns;  // pipeline wait limit (0: the default; a test limit otherwise)
  const void* residual;  // NM == 1: added to y (y's dtype), or nullptr
  const void* rms_w;     // NM == 1: RMSNorm weights (x's dtype), or nullptr
  float eps;
};

// 8 consecutive elements of x (or of the RMSNorm weights) as fp32 (16-byte aligned)
template <bool XB>
__device__ __forceinline__ void load8(const void* p, int e0, float (&v)[8]) {
  if constexpr (XB) {
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + e0);
    const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else {
    const float* q = reinterpret_cast<const float*>(p) + e0;
    const float4 a = *reinterpret_cast<const float4*>(q);
    const float4 b = *reinterpret_cast<const float4*>(q + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Digit d of four integers, element b in byte b.
__device__ __forceinline__ uint32_t digit_word(const int (&X)[8], int o, int d) {
  const uint32_t sel = uint32_t(d) | (uint32_t(d + 4) << 4);
  const uint32_t lo = __byte_perm(uint32_t(X[o]), uint32_t(X[o + 1]), sel);
  const uint32_t hi = __byte_perm(uint32_t(X[o + 2]), uint32_t(X[o + 3]), sel);
  return __byte_perm(lo, hi, 0x5410);
}

// The records of group `grp` from the 8 elements v of lane L (= lane % 16) of
// a half warp: elements 8L..8L+7, i.e. shift class t = L / 4 and bytes
// 8(L%4)..8(L%4)+7 = words 2(L%4), 2(L%4)+1 of the group.  Whole warp (the
// two halves take two groups); `active` false for a half without a group.
template <int D>
__device__ __forceinline__ void group_records(const float (&v)[8], bool active, int grp, uint32_t* rec, int lane) {
  using C = Slot<D>;
  const int L = lane & 15, t = L >> 2, j0 = 2 * (L & 3);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int F = m > 0.f ? (8 * D - 1) - exponent_of(m) : 0;
  const int fa = F / 2, fb = F - fa;  // x * 2^F as two exact power-of-two multiplies
  const float sA = exp2i(fa), sB = exp2i(fb);
  constexpr int kLim = int((1u << (8 * D - 1)) - 1u);
  int X[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) X[i] = max(-kLim, min(kLim, __float2int_rn(__fmul_rn(__fmul_rn(v[i], sA), sB))));
  const int slot = grp * C::kPerGroup + j0 / C::W;  // both words of this lane lie in one slot
  uint32_t* r = rec + size_t(slot) * C::kStride;
  int sums[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const uint32_t w0 = digit_word(X, 0, d), w1 = digit_word(X, 4, d);
    const int jj = j0 % C::W;
    if (active) {
      r[(jj * 4 + t) * D + d] = w0;
      r[((jj + 1) * 4 + t) * D + d] = w1;
    }
    sums[d] = d == D - 1 ? dp4a_us(0x01010101u, w0, dp4a_us(0x01010101u, w1, 0))
                         : dp4a_uu(0x01010101u, w0, dp4a_uu(0x01010101u, w1, 0));
  }
  // the slot's digit sums: the lanes of one slot differ in t (bits 2, 3 of L)
  // and, for four-word slots, in bit 0
#pragma unroll
  for (int d = 0; d < D; ++d) {
    if constexpr (C::W == 4) sums[d] += __shfl_xor_sync(0xffffffffu, sums[d], 1);
    sums[d] += __shfl_xor_sync(0xffffffffu, sums[d], 4);
    sums[d] += __shfl_xor_sync(0xffffffffu, sums[d], 8);
  }
  if (active && t == 0 && (C::W == 2 || (L & 1) == 0)) {
    int* ri = reinterpret_cast<int*>(r + C::kDig);
#pragma unroll
    for (int d = 0; d < D; ++d) ri[d] = sums[d];
    reinterpret_cast<float*>(r + C::kDig)[D] = exp2i(-fa);
    reinterpret_cast<float*>(r + C::kDig)[D + 1] = exp2i(-fb);
  }
}

// sum_k w_k X_k over one slot of one row (scaled by 2^-F): `wd` holds the
// row's W code words of the slot, `xd` the slot's digits, `S` its digit sums.
template <int D>
__device__ __forceinline__ float slot_dot(const uint32_t (&wd)[Slot<D>::W], const uint32_t (&xd)[Slot<D>::kDig],
                                         const int (&S)[D], float fa, float fb) {
  using C = Slot<D>;
  int aA[D], aB[D];  // classes t = 2, 3 (codes) and t = 0, 1 (16 x codes), per digit
#pragma unroll
  for (int d = 0; d < D; ++d) aA[d] = aB[d] = 0;
#pragma unroll
  for (int jj = 0; jj < C::W; ++jj) {
    const uint32_t w = wd[jj], w2 = w >> 2;
    const uint32_t m3 = w & 0x03030303u, m2 = w2 & 0x03030303u;  // t = 3, t = 2
    const uint32_t m1 = w & 0x30303030u, m0 = w2 & 0x30303030u;  // t = 1, t = 0 (x 16)
    const uint32_t* x = xd + jj * 4 * D;                         // [t][d]
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (d == D - 1) {  // signed top digit
        aA[d] = dp4a_us(m3, x[3 * D + d], dp4a_us(m2, x[2 * D + d], aA[d]));
        aB[d] = dp4a_us(m1, x[1 * D + d], dp4a_us(m0, x[0 * D + d], aB[d]));
      } else {
        aA[d] = dp4a_uu(m3, x[3 * D + d], dp4a_uu(m2, x[2 * D + d], aA[d]));
        aB[d] = dp4a_uu(m1, x[1 * D + d], dp4a_uu(m0, x[0 * D + d], aB[d]));
      }
    }
  }
  float p;
  if constexpr (D <= 3) {  // |sum| < 2^29: exact in int32
    int v = 0;
#pragma unroll
    for (int d = D - 1; d >= 0; --d) v = v * 256 + (aA[d] + (aB[d] >> 4) - S[d]);  // aB is a multiple of 16
    p = float(v);  // exact: |v| < 2^24 for D = 2; for D = 3 rounded once
  } else {
    p = 0.f;
#pragma unroll
    for (int d = D - 1; d >= 0; --d) p = p * 256.f + float(aA[d] + (aB[d] >> 4) - S[d]);
  }
  return (p * fa) * fb;
}

// named barrier 1: arrive without waiting / wait for n threads in all
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <bool YB>
__device__ __forceinline__ void store_out(void* y, int row, float v) {
  if (YB)
    reinterpret_cast<uint16_t*>(y)[row] = f32_to_bf16_bits_rn(v);
  else
    reinterpret_cast<float*>(y)[row] = v;
}

// NM = 1: y = scale * W x (+ residual; RMSNorm of x first when rms_w is set).
// NM = 2: h = max(0, scale_g W_g x)^2 * (scale_u W_u x).
template <int D, bool XB, bool YB, int NM>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_i2s_slot_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ packed2,
                         const void* __restrict__ x, void* __restrict__ y, SGeom g) {
  using C = Slot<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t wbar;
  __shared__ int abort_flag;
  __shared__ float red[kWarps];
  __shared__ float tscale[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = g.ks == 2 ? int(cluster_ctarank()) : 0;
  const int c = blockIdx.x / g.ks;
  const int r0 = c * g.q + min(c, g.rem);
  const int rows = g.q + (c < g.rem ? 1 : 0);
  const int R = NM * rows;  // rows in shared memory: matrix m's row i at m * rows + i
  const int64_t row_bytes = g.K / 4;
  const int gx0 = rank * g.nC;  // first group of this CTA's share of K
  uint32_t* rec = reinterpret_cast<uint32_t*>(smem + g.off_rec);
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  auto pk = [&](int m) { return (NM == 2 && m) ? packed2 : packed; };

  if (tid == 0) {
    mbar_init(&wbar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&wbar, uint32_t(R) * uint32_t(g.RS));
    abort_flag = 0;
  }
  __syncthreads();
  if (tid < NM)  // the tensor scales (after the codes): fetched now, not on the epilogue's critical path
    tscale[tid] = *reinterpret_cast<const float*>(pk(tid) + int64_t(g.N) * row_bytes);
  for (int t = tid; t < R; t += kThreads) {
    const int m = t / rows, i = t - m * rows;
    bulk_g2s(smem + size_t(t) * g.RS, pk(m) + int64_t(r0 + i) * row_bytes + 32 * gx0, uint32_t(g.RS), &wbar,
             policy_evict_first());
  }
  // the next kernel's CTAs may become resident now: they fetch their own
  // weights, then wait for this grid to complete before reading its output
  pdl_launch_dependents();
  pdl_wait();

  // ---- activation records ----------------------------------------------------
  const void* rmsw = NM == 1 ? g.rms_w : nullptr;
  float rinv = 1.f;
  if (rmsw) {
    // RMSNorm factor 1 / sqrt(mean(x^2) + eps); every CTA adds in the same order
    float ss = 0.f;
    for (int e = 8 * tid; e < g.K; e += 8 * kThreads) {
      float v[8];
      load8<XB>(x, e, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(v[i], v[i]));
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot = __fadd_rn(tot, red[w]);
    rinv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, float(g.K)), g.eps)));
  }
  // two groups per warp and pass; the next pass's elements are loaded before
  // this pass is converted, so only the first load's latency is exposed
  const int L = lane & 15;
  float v[8], wv[8];
  auto fetch = [&](int gb, float (&a)[8], float (&b)[8]) {
    const int grp = gb + (lane >> 4);
    if (gb < g.nC && grp < g.nC) {
      load8<XB>(x, (gx0 + grp) * 128 + 8 * L, a);
      if (rmsw) load8<XB>(rmsw, (gx0 + grp) * 128 + 8 * L, b);
    }
  };
  fetch(2 * warp, v, wv);
  for (int gb = 2 * warp; gb < g.nC; gb += 2 * kWarps) {
    float vn[8], wn[8];
    fetch(gb + 2 * kWarps, vn, wn);
    const int grp = gb + (lane >> 4);
    const bool active = grp < g.nC;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!active) v[i] = 0.f;
      else if (rmsw) v[i] = __fmul_rn(__fmul_rn(v[i], rinv), wv[i]);
    }
    group_records<D>(v, active, grp, rec, lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = vn[i];
      wv[i] = wn[i];
    }
  }
  __syncthreads();
  const float sc0 = tscale[0], sc1 = tscale[NM - 1];

  // ---- slot dot products -------------------------------------------------------
  bool waited = false;
  // With g.ovl (fused gate/up, a whole warp without a slot) the rows of the
  // first h1 outputs -- gate rows [0, h1) and up rows [rows, rows + h1) --
  // come first; the last warp waits for them at a named barrier and sums
  // those outputs while the other warps compute the remaining rows.
  const int h1 = (NM == 2 && g.ovl) ? rows / 2 : 0;
  if (h1 > 0) {
    if (warp < kWarps - 1) {
      const bool has = tid < g.NS * g.nl;  // one slot at most (NS * nl <= 480)
      const int s = tid % g.NS, j = tid / g.NS;
      uint32_t xd[C::kDig];
      int S[D];
      float fa = 0.f, fb = 0.f;
      if (has) {
        const uint32_t* r = rec + size_t(s) * C::kStride;
#pragma unroll
        for (int k = 0; k < C::kDig / 4; ++k) {
          const uint4 q = *reinterpret_cast<const uint4*>(r + 4 * k);
          xd[4 * k] = q.x; xd[4 * k + 1] = q.y; xd[4 * k + 2] = q.z; xd[4 * k + 3] = q.w;
        }
#pragma unroll
        for (int d = 0; d < D; ++d) S[d] = reinterpret_cast<const int*>(r + C::kDig)[d];
        fa = reinterpret_cast<const float*>(r + C::kDig)[D];
        fb = reinterpret_cast<const float*>(r + C::kDig)[D + 1];
        if (!abort_flag && !mbar_wait_limited(&wbar, 0, g.err, g.wait_ns)) abort_flag = 1;
      }
      const bool go = has && !abort_flag;
      const uint8_t* wp = smem + size_t(s) * (4 * C::W);
      auto do_row = [&](int row) {
        uint32_t wd[C::W];
        if constexpr (C::W == 4) {
          const uint4 q = *reinterpret_cast<const uint4*>(wp + size_t(row) * g.RS);
          wd[0] = q.x; wd[1] = q.y; wd[2] = q.z; wd[3] = q.w;
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(wp + size_t(row) * g.RS);
          wd[0] = q.x; wd[1] = q.y;
        }
        part[size_t(row) * g.PS + s] = slot_dot<D>(wd, xd, S, fa, fb);
      };
      const int hh = rows - h1;
      int v = j;  // processing order: gate/up rows of outputs [0, h1), then of [h1, rows)
      if (go) {
#pragma unroll 1
        for (; v < 2 * h1; v += g.nl) do_row(v < h1 ? v : rows + (v - h1));
      }
      named_arrive(1, kThreads);  // every thread of warps 0 .. kWarps-2, on every path
      if (go) {
#pragma unroll 1
        for (; v < R; v += g.nl) {
          const int u = v - 2 * h1;
          do_row(u < hh ? h1 + u : rows + h1 + (u - hh));
        }
      }
    } else {
      named_sync(1, kThreads);
      if constexpr (NM == 2) {
        if (!abort_flag) {
          for (int o = lane; o < h1; o += 32) {
            const float* pg = part + size_t(o) * g.PS;
            const float* pu = part + size_t(rows + o) * g.PS;
            float a = 0.f, b = 0.f;
            int s0 = 0;
            for (; s0 + 3 < g.NS; s0 += 4) {
              const float t0 = pg[s0], t1 = pg[s0 + 1], t2 = pg[s0 + 2], t3 = pg[s0 + 3];
              const float u0 = pu[s0], u1 = pu[s0 + 1], u2 = pu[s0 + 2], u3 = pu[s0 + 3];
              a += t0; a += t1; a += t2; a += t3;
              b += u0; b += u1; b += u2; b += u3;
            }
            for (; s0 < g.NS; ++s0) {
              a += pg[s0];
              b += pu[s0];
            }
            const float gv = fmaxf(a * sc0, 0.f), uv = b * sc1;
            store_out<YB>(y, r0 + o, (gv * gv) * uv);
          }
        }
      }
    }
  } else {
    for (int vs = tid; vs < g.NS * g.nl; vs += kThreads) {
      const int s = vs % g.NS, j = vs / g.NS;
      uint32_t xd[C::kDig];
      const uint32_t* r = rec + size_t(s) * C::kStride;
#pragma unroll
      for (int k = 0; k < C::kDig / 4; ++k) {
        const uint4 q = *reinterpret_cast<const uint4*>(r + 4 * k);
        xd[4 * k] = q.x; xd[4 * k + 1] = q.y; xd[4 * k + 2] = q.z; xd[4 * k + 3] = q.w;
      }
      int S[D];
#pragma unroll
      for (int d = 0; d < D; ++d) S[d] = reinterpret_cast<const int*>(r + C::kDig)[d];
      const float fa = reinterpret_cast<const float*>(r + C::kDig)[D];
      const float fb = reinterpret_cast<const float*>(r + C::kDig)[D + 1];
      if (!waited) {
        waited = true;
        if (!abort_flag && !mbar_wait_limited(&wbar, 0, g.err, g.wait_ns)) abort_flag = 1;
      }
      if (abort_flag) break;
      const uint8_t* wp = smem + size_t(s) * (4 * C::W);
#pragma unroll 1
      for (int row = j; row < R; row += g.nl) {
        uint32_t wd[C::W];
        if constexpr (C::W == 4) {
          const uint4 q = *reinterpret_cast<const uint4*>(wp + size_t(row) * g.RS);
          wd[0] = q.x; wd[1] = q.y; wd[2] = q.z; wd[3] = q.w;
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(wp + size_t(row) * g.RS);
          wd[0] = q.x; wd[1] = q.y;
        }
        part[size_t(row) * g.PS + s] = slot_dot<D>(wd, xd, S, fa, fb);
      }
    }
  }
  __syncthreads();

  // ---- the partials of each row in slot order: tpr threads per row (slots
  //      tpr apart, in order), then a fixed butterfly; lane 0 of the row keeps
  //      the result, so it does not depend on timing ------------------------------
  if (!abort_flag) {
    const int per_out = NM * g.tpr;         // threads per output
    const int opw = 32 / per_out;           // outputs per warp and pass
    const int sub = lane % per_out, m = sub / g.tpr, l = sub % g.tpr;
    for (int ob = h1 + warp * opw; ob < rows; ob += kWarps * opw) {
      const int o = ob + lane / per_out;
      float a = 0.f;
      if (o < rows) {
        // up to 16 partials in flight, added in slot order
        const float* pr = part + size_t(m * rows + o) * g.PS;
        int s0 = l;
        for (; s0 + 3 * g.tpr < g.NS; s0 += 4 * g.tpr) {
          float t[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) t[k] = pr[s0 + k * g.tpr];
#pragma unroll
          for (int k = 0; k < 4; ++k) a += t[k];
        }
        for (; s0 < g.NS; s0 += g.tpr) a += pr[s0];
      }
      for (int off = g.tpr >> 1; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      const float b = NM == 2 ? __shfl_down_sync(0xffffffffu, a, g.tpr) : 0.f;  // the up row's sum
      if (g.ks == 2) {
        if (o < rows && sub == 0) reinterpret_cast<float*>(smem + g.off_sum)[o] = a;  // this CTA's share
      } else if (o < rows && sub == 0) {
        const int row = r0 + o;
        if (NM == 2) {
          const float gv = fmaxf(a * sc0, 0.f), uv = b * sc1;
          store_out<YB>(y, row, (gv * gv) * uv);
        } else {
          float out = a * sc0;
          if (g.residual)
            out += YB ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(g.residual)[row])
                      : reinterpret_cast<const float*>(g.residual)[row];
          store_out<YB>(y, row, out);
        }
      }
    }
  } else if (tid == 0) {
    mbar_wait_bounded(&wbar, 0, nullptr);  // let the copies still in flight land before the CTA exits
  }
  if (g.ks == 2) {
    // the two CTAs' shares of each row, added in rank order; rank r finishes
    // half of the rows.  Every thread of both CTAs reaches both cluster
    // barriers, whatever happened before (the second keeps this CTA's shares
    // readable until the peer is done).
    cluster_sync();
    if (NM == 1 && !abort_flag) {
      const float* sum = reinterpret_cast<const float*>(smem + g.off_sum);
      const int half = (rows + 1) / 2;
      for (int o = rank * half + tid; o < min(rows, (rank + 1) * half); o += kThreads) {
        const float mine = sum[o], peer = ld_peer_f32(sum + o, uint32_t(rank ^ 1));
        const float a = rank == 0 ? mine + peer : peer + mine;
        const int row = r0 + o;
        float out = a * sc0;
        if (g.residual)
          out += YB ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(g.residual)[row])
                    : reinterpret_cast<const float*>(g.residual)[row];
        store_out<YB>(y, row, out);
      }
    }
    cluster_sync();
  }
}

template <int D, int NM>
bool plan_slot(SGeom& g, int64_t N, int64_t K, int max_smem, int nsm, int ks) {
  using C = Slot<D>;
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  if ((K / 128) % ks || (ks > 1 && NM != 1)) return false;
  g.N = int(N);
  g.K = int(K);
  g.ks = ks;
  g.nC = int(K / 128) / ks;
  g.NS = g.nC * C::kPerGroup;
  const int clusters = int(std::min<int64_t>(nsm / ks, N));
  g.grid = clusters * ks;
  g.q = g.N / clusters;
  g.rem = g.N % clusters;
  g.nl = std::max(1, kThreads / g.NS);
  g.PS = g.NS | 1;
  g.RS = 32 * g.nC;
  const int rows_max = g.q + (g.rem ? 1 : 0);
  // threads per row for the final sums: as many as fit one pass over the rows, at most NS
  g.ovl = (NM == 2 && g.NS * g.nl <= kThreads - 32 && rows_max >= 2) ? 1 : 0;
  g.tpr = 32 / NM;
  while (g.tpr > 1 && ((kThreads / (NM * g.tpr)) < rows_max || g.tpr > g.NS)) g.tpr >>= 1;
  const uint64_t R = uint64_t(NM) * rows_max;
  const uint64_t off_rec = up(R * uint64_t(g.RS), 128);
  const uint64_t off_part = up(off_rec + 4ull * g.NS * C::kStride, 128);
  const uint64_t off_sum = up(off_part + 4ull * R * g.PS, 16);
  const uint64_t total = off_sum + (ks > 1 ? 4ull * rows_max : 0);
  if (total > uint64_t(max_smem)) return false;
  g.off_rec = uint32_t(off_rec);
  g.off_part = uint32_t(off_part);
  g.off_sum = uint32_t(off_sum);
  g.smem = uint32_t(total);
  return true;
}

struct SPlan {
  SGeom g;
  bool ok;
};

template <int D, bool XB, bool YB, int NM>
cudaError_t run_slot(const uint8_t* packed, const uint8_t* packed2, const void* x, void* y, int64_t N, int64_t K,
                     cudaStream_t st, const void* residual, const void* rms_w, float eps) {
  auto kern = gemv_i2s_slot_kernel<D, XB, YB, NM>;
  static PlanCache<SPlan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  SPlan p{};
  if (!cache.get(dev, N, K, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int cap = max_optin - 1024;  // static shared memory of the kernel stays below 1 KB
    // a long K is split over a cluster of two CTAs (each builds half of the
    // records and takes half of every row); prefer plans that leave room for
    // the next launch's CTA on the SM
    const int nsm = sm_count(), co = std::min(cap, kCoResident);
    const bool split = NM == 1 && K / 128 >= 40;
    p.ok = (split && plan_slot<D, NM>(p.g, N, K, co, nsm, 2)) || plan_slot<D, NM>(p.g, N, K, co, nsm, 1) ||
           (split && plan_slot<D, NM>(p.g, N, K, cap, nsm, 2)) || plan_slot<D, NM>(p.g, N, K, cap, nsm, 1);
    if (p.ok) {
      cudaError_t e = raise_smem_cap(kern, dev, cap);
      if (e != cudaSuccess) return e;
      p.g.err = dev_error_ptr();
    }
    cache.put(dev, N, K, p);
  }
  if (!p.ok || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(rms_w) & 15))
    return cudaErrorNotSupported;
  p.g.wait_ns = wait_limit_ns();
  p.g.residual = residual;
  p.g.rms_w = rms_w;
  p.g.eps = eps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.g.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.g.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (overlap_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (p.g.ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = unsigned(p.g.ks);
    attr[na].val.clusterDim.y = 1;
    attr[na++].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, packed, packed2, x, y, p.g);
}

}  // namespace

// cudaErrorNotSupported: no plan here (the CTA's rows, the records and the
// partials exceed shared memory, or x / rms_w is not 16-byte aligned);
// nothing was launched.
cudaError_t launch_gemv_i2s_slot(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N,
                                 int64_t K, cudaStream_t s, const void* residual, const void* rms_w, float eps) {
  const bool xb = xt == BL_BF16, yb = yt == BL_BF16;
  if (xb)
    return yb ? run_slot<2, true, true, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps)
              : run_slot<3, true, false, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps);
  return yb ? run_slot<3, false, true, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps)
            : run_slot<3, false, false, 1>(packed, packed, x, y, N, K, s, residual, rms_w, eps);
}

cudaError_t launch_gemv_i2s_gate_up_slot(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x,
                                         bl_dtype xt, void* h, bl_dtype ht, int64_t N, int64_t K, cudaStream_t s) {
  const bool xb = xt == BL_BF16, hb = ht == BL_BF16;
  if (xb)
    return hb ? run_slot<2, true, true, 2>(packed_gate, packed_up, x, h, N, K, s, nullptr, nullptr, 0.f)
              : run_slot<3, true, false, 2>(packed_gate, packed_up, x, h, N, K, s, nullptr, nullptr, 0.f);
  return hb ? run_slot<3, false, true, 2>(packed_gate, packed_up, x, h, N, K, s, nullptr, nullptr, 0.f)
            : run_slot<3, false, false, 2>(packed_gate, packed_up, x, h, N, K, s, nullptr, nullptr, 0.f);
}

}  // namespace bl
