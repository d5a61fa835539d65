// W1A8 product for one token, activation-stationary ("binary-gemm" card,
// sections "API" binary_gemm and "Method"):
//   dot[n,g] = sum_{k in g} w[n,k] q[k] = 2 * sum_{k in g, bit 1} q[k] - sum_{k in g} q[k]   (exact)
//   y[n]     = bf16( s * sum_g ws[n,g] * dot[n,g] + bias[n] )
// for 128-element groups.
//
// Every thread owns one group (a slot): the group's activations, rearranged
// once per CTA into 32 words -- word w, bit class j holds q[32w + j + 8b] in
// byte b -- sit in its registers, and rows stream through it.  For a row,
// one 16-byte shared-memory load brings the group's four bit words; per word
// and class the mask  word & (0x01010101 << j)  holds the bits of elements
// j, j+8, j+16, j+24 (one per byte, times 2^j), so one dp4a adds 2^j times
// their activations.  The eight class sums are kept apart and combined once
// per row and group: acc_j = 2^j S_j, so T = sum_j acc_j 2^(7-j) = 2^7 sum_j
// S_j exactly, by multiply-adds with runtime powers of two (they stay on the
// FMA pipe; the ALU pipe carries the masks); then scaled by the row's fp16
// group scale and written as the row's partial.  The threads of a slot take
// rows j, j + nl, ... (nl threads per slot).
//
// Streaming.  A CTA takes a contiguous range of tiles of RT rows; a tile's
// bits and group scales are contiguous in memory and arrive by two bulk
// copies into a ring of stages.  After a tile's products the CTA meets once,
// and the stage goes back to the copy engine.  When a whole warp holds no
// slot, that warp sums the rows of the previous tile (a lane per row, the
// slots in order) while the others compute the current one; otherwise all
// warps sum the tile's rows after the barrier (tpr threads per row over the
// slots in order, then a fixed butterfly).  Either way the other partials
// buffer takes the next tile's products.
//
// Fused activation quantization (XQ != 0): each CTA quantizes the token
// itself with act_quant.cuh's binary32 steps, so codes and scale equal the
// stand-alone kernel's bit for bit.
#include <algorithm>

#include "act_quant.cuh"
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRecWords = 36;  // 32 activation words, the group's sum of q, padding (16-byte records)
constexpr int kRowsPerThread = 10;  // rows of a tile per thread

struct Geom {
  int N, K, nG;         // rows, columns, groups per row (= slots)
  int nl, RT, PS, tpr;  // threads per slot, rows per tile, partials per row (odd), threads per row in the sums
  int ntiles, stages;
  int one;              // 1 (a runtime value)
  int rw;               // 1: the last warp has no slot and sums the rows (one tile behind)
  uint32_t rb, sb;      // bit bytes and scale bytes of a row
  uint32_t stage_bytes, off_bar, off_stage, off_part, off_rec, off_q, smem;
  unsigned int* err;
};

template <bool DOTS, int XQ>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_w1a8_m1_kernel(const int8_t* __restrict__ q, const float* __restrict__ s, const void* __restrict__ x,
                        const uint8_t* __restrict__ wq, const uint8_t* __restrict__ ws,
                        const uint16_t* __restrict__ bias, uint16_t* __restrict__ y, int32_t* __restrict__ dots,
                        Geom g) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  uint64_t* qbar = full + g.stages;
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  uint32_t* rec = reinterpret_cast<uint32_t*>(smem + g.off_rec);
  int8_t* qs = reinterpret_cast<int8_t*>(smem + g.off_q);
  __shared__ int abort_flag;
  __shared__ float tok_scale, tok_inv;
  __shared__ float red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // contiguous tile range of this CTA
  const int t_begin = int(int64_t(blockIdx.x) * g.ntiles / gridDim.x);
  const int t_end = int(int64_t(blockIdx.x + 1) * g.ntiles / gridDim.x);
  const int my_tiles = t_end - t_begin;
  auto issue = [&](int i) {  // tile t_begin + i into stage i % stages (one thread)
    const int t = t_begin + i, st = i % g.stages;
    const int r0 = t * g.RT, nr = min(g.RT, g.N - r0);
    uint8_t* dst = smem + g.off_stage + size_t(st) * g.stage_bytes;
    mbar_arrive_expect_tx(&full[st], uint32_t(nr) * (g.rb + g.sb));
    const uint64_t pol = policy_evict_first();
    bulk_g2s(dst, wq + int64_t(r0) * g.rb, uint32_t(nr) * g.rb, &full[st], pol);
    bulk_g2s(dst + size_t(g.RT) * g.rb, ws + int64_t(r0) * g.sb, uint32_t(nr) * g.sb, &full[st], pol);
  };

  int issued = 0;  // thread 0: tiles whose copies were issued
  if (tid == 0) {
    for (int st = 0; st < g.stages; ++st) mbar_init(&full[st], 1);
    mbar_init(qbar, 1);
    abort_flag = 0;
    fence_barrier_init();
    for (; issued < min(my_tiles, g.stages); ++issued) issue(issued);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  // ---- the token: codes into shared memory, then the group records ----------
  float scale;
  if (XQ == 0) {
    if (tid == 0) {
      mbar_arrive_expect_tx(qbar, uint32_t(g.K));
      bulk_g2s(qs, q, uint32_t(g.K), qbar, policy_evict_first());
    }
    scale = s[0];
    if (!mbar_wait_bounded(qbar, 0, g.err)) abort_flag = 1;
  } else {
    token_scales<1, XQ == 2>(x, g.K, red, &tok_scale, &tok_inv);  // ends with a CTA barrier
    const float iv = tok_inv;
    for (int i = tid; i < g.K / 8; i += kThreads) {
      float v[8];
      load8<XQ == 2>(x, i, v);
      reinterpret_cast<uint2*>(qs)[i] = quant8(v, iv);
    }
    scale = tok_scale;
  }
  __syncthreads();
  for (int e = tid; e < g.nG * 32; e += kThreads) {
    const int c = e >> 5, w = (e >> 3) & 3, j = e & 7;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(qs) + 128 * c + 32 * w + j;
    rec[c * kRecWords + w * 8 + j] =
        uint32_t(src[0]) | (uint32_t(src[8]) << 8) | (uint32_t(src[16]) << 16) | (uint32_t(src[24]) << 24);
  }
  for (int c = warp; c < g.nG; c += kWarps) {  // sum of the group's codes
    const int v = dp4a_us(0x01010101u, reinterpret_cast<const uint32_t*>(qs + 128 * c)[lane], 0);
    const int tot = redux_add(v);
    if (lane == 0) reinterpret_cast<int*>(rec)[c * kRecWords + 32] = tot;
  }
  __syncthreads();

  // ---- this thread's slot ------------------------------------------------------
  const int slot = tid % g.nG, j0 = tid / g.nG;
  // 2^(7-j) as runtime values, so that the class combine stays multiply-adds
  int p2[7];
#pragma unroll
  for (int jc = 0; jc < 7; ++jc) p2[jc] = g.one << (7 - jc);
  const bool has_slot = tid < g.nG * g.nl;
  uint32_t xa[32];
  int qsum = 0;
  if (has_slot) {
    const uint32_t* r = rec + slot * kRecWords;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(r + 4 * k);
      xa[4 * k] = v.x; xa[4 * k + 1] = v.y; xa[4 * k + 2] = v.z; xa[4 * k + 3] = v.w;
    }
    qsum = reinterpret_cast<const int*>(r)[32];
  }

  const int per_out = g.tpr, opw = 32 / per_out, l = lane % per_out;
  const bool rwarp = g.rw && warp == kWarps - 1;  // this warp sums rows while the others compute
  for (int i = 0; i <= my_tiles; ++i) {
    if (i < my_tiles && !rwarp) {
      const int st = i % g.stages, t = t_begin + i;
      const int r0 = t * g.RT, nr = min(g.RT, g.N - r0);
      float* pb = part + size_t(i & 1) * g.RT * g.PS;
      if (!abort_flag && !mbar_wait_bounded(&full[st], uint32_t(i / g.stages) & 1u, g.err)) abort_flag = 1;
      const uint8_t* stage = smem + g.off_stage + size_t(st) * g.stage_bytes;
      if (has_slot && !abort_flag && j0 < nr) {
        // the next row's bit words are loaded while this row's are decoded
        uint4 wn = *reinterpret_cast<const uint4*>(stage + size_t(j0) * g.rb + 16 * slot);
#pragma unroll 1
        for (int row = j0; row < nr; row += g.nl) {
          const uint4 wv = wn;
          if (row + g.nl < nr) wn = *reinterpret_cast<const uint4*>(stage + size_t(row + g.nl) * g.rb + 16 * slot);
          const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
          int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
          for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) acc[jc] = dp4a_us(wd[w] & (0x01010101u << jc), xa[8 * w + jc], acc[jc]);
          // acc_j = 2^j S_j, so T = sum_j acc_j 2^(7-j) = 2^7 sum_j S_j (|T| < 2^21)
          int T = acc[7];
#pragma unroll
          for (int jc = 6; jc >= 0; --jc) T += acc[jc] * p2[jc];
          const int dot = (T >> 6) - qsum;
          if (DOTS) dots[int64_t(r0 + row) * g.nG + slot] = dot;
          const float wsf = __half2float(__ushort_as_half(
              *reinterpret_cast<const uint16_t*>(stage + size_t(g.RT) * g.rb + size_t(row) * g.sb + 2 * slot)));
          pb[row * g.PS + slot] = wsf * float(dot);
        }
      }
    }
    if (rwarp && i >= 1 && !abort_flag) {  // the rows of tile i - 1, one lane per row, slots in order
      const int k = i - 1, r0 = (t_begin + k) * g.RT, nr = min(g.RT, g.N - r0);
      const float* pb = part + size_t(k & 1) * g.RT * g.PS;
      for (int o = lane; o < nr; o += 32) {
        const float* pr = pb + o * g.PS;
        float a = 0.f;
        int s0 = 0;
        for (; s0 + 3 < g.nG; s0 += 4) {
          const float t0 = pr[s0], t1 = pr[s0 + 1], t2 = pr[s0 + 2], t3 = pr[s0 + 3];
          a += t0; a += t1; a += t2; a += t3;
        }
        for (; s0 < g.nG; ++s0) a += pr[s0];
        float val = a * scale;
        if (bias) val += bf16_bits_to_f32(bias[r0 + o]);
        y[r0 + o] = f32_to_bf16_bits_rn(val);
      }
    }
    __syncthreads();  // tile i's partials are complete, its stage is free, tile i - 1's rows are summed
    if (i < my_tiles) {
      if (tid == 0 && i + g.stages < my_tiles && !abort_flag) issue(issued++);
      if (!g.rw) {
        const int t = t_begin + i, r0 = t * g.RT, nr = min(g.RT, g.N - r0);
        const float* pb = part + size_t(i & 1) * g.RT * g.PS;
        // the tile's rows: tpr threads per row over the slots in order, then a butterfly
        if (!abort_flag)
          for (int ob = warp * opw; ob < nr; ob += kWarps * opw) {
            const int o = ob + lane / per_out;
            float a = 0.f;
            if (o < nr)
            {
              const float* pr = pb + o * g.PS;
              int s0 = l;
              for (; s0 + 3 * per_out < g.nG; s0 += 4 * per_out) {
                const float t0 = pr[s0], t1 = pr[s0 + per_out], t2 = pr[s0 + 2 * per_out], t3 = pr[s0 + 3 * per_out];
                a += t0; a += t1; a += t2; a += t3;
              }
              for (; s0 < g.nG; s0 += per_out) a += pr[s0];
            }
            for (int off = per_out >> 1; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (o < nr && l == 0) {
              float val = a * scale;
              if (bias) val += bf16_bits_to_f32(bias[r0 + o]);
              y[r0 + o] = f32_to_bf16_bits_rn(val);
            }
          }
      }
    }
  }
  if (abort_flag && tid == 0) {
    // let copies still in flight land before the CTA exits
    for (int k = max(0, issued - g.stages); k < issued; ++k)
      mbar_wait_bounded(&full[k % g.stages], uint32_t(k / g.stages) & 1u, nullptr);
    if (XQ == 0) mbar_wait_bounded(qbar, 0, nullptr);
  }
}

bool plan(Geom& g, int64_t N, int64_t K, int max_smem, int nsm) {
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.N = int(N);
  g.K = int(K);
  g.nG = int(K / 128);
  if (g.nG > kThreads) return false;
  g.nl = kThreads / g.nG;
  // kRowsPerThread rows per thread and tile, rounded up to a multiple of 8 so that every
  // tile's scales start on a 16-byte boundary (nG * RT * 2 % 16 == 0)
  g.RT = int(std::min<int64_t>((int64_t(g.nl) * kRowsPerThread + 7) / 8 * 8, 4096));
  g.PS = g.nG | 1;
  g.rb = uint32_t(K / 8);
  g.sb = uint32_t(g.nG * 2);
  g.tpr = 32;
  while (g.tpr > 1 && ((kThreads / g.tpr) < g.RT || g.tpr > g.nG)) g.tpr >>= 1;
  g.ntiles = int((N + g.RT - 1) / g.RT);
  g.one = 1;
  g.rw = g.nG * g.nl <= kThreads - 32 ? 1 : 0;
  g.stage_bytes = uint32_t(up(uint64_t(g.RT) * (g.rb + g.sb), 128));
  for (int st = 4; st >= 2; --st) {
    uint64_t off = 0;
    g.off_bar = uint32_t(off);
    off = up(off + 8ull * (st + 1), 128);
    g.off_stage = uint32_t(off);
    off += uint64_t(st) * g.stage_bytes;
    g.off_part = uint32_t(off);
    off = up(off + 4ull * 2 * g.RT * g.PS, 128);
    g.off_rec = uint32_t(off);
    off = up(off + 4ull * g.nG * kRecWords, 128);
    g.off_q = uint32_t(off);
    off = up(off + uint64_t(K), 128);
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
  int grid;
  bool ok;
};

template <bool DOTS, int XQ>
cudaError_t run(const int8_t* q, const float* s, const void* x, const int32_t* wq, const uint16_t* ws,
                const uint16_t* bias, int64_t N, int64_t K, uint16_t* y, int32_t* dots, cudaStream_t st) {
  auto kern = gemm_w1a8_m1_kernel<DOTS, XQ>;
  static PlanCache<Plan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  Plan p{};
  if (!cache.get(dev, N, K, &p)) {
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    const int budget = max_optin - int(fa.sharedSizeBytes);
    p.ok = plan(p.g, N, K, budget, sm_count());
    if (p.ok) {
      e = raise_smem_cap(kern, dev, budget);
      if (e != cudaSuccess) return e;
      p.grid = std::min(p.g.ntiles, sm_count());
      p.g.err = dev_error_ptr();
    }
    cache.put(dev, N, K, p);
  }
  if (!p.ok) return cudaErrorNotSupported;
  return launch(kern, dim3(p.grid), dim3(kThreads), p.g.smem, st, overlap_enabled(), q, s, x,
                reinterpret_cast<const uint8_t*>(wq), reinterpret_cast<const uint8_t*>(ws), bias, y, dots, p.g);
}

}  // namespace

// One token, 128-element groups, whole tiles of bits and scales 16-byte aligned.
bool w1a8_m1_applicable(int64_t M, int64_t N, int64_t K, int G) {
  return M == 1 && G == 128 && K % 128 == 0 && K / 128 <= kThreads && (N * (K / 128)) % 8 == 0;
}

cudaError_t launch_gemm_w1a8_m1(const int8_t* q, const float* s, const void* x, bl_dtype xt, const int32_t* wq,
                                const uint16_t* ws, const uint16_t* bias, int64_t N, int64_t K, uint16_t* y,
                                int32_t* dots, cudaStream_t st) {
  if (x) {  // quantized here (rows 16-byte aligned)
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0) return cudaErrorNotSupported;
    return xt == BL_BF16 ? run<false, 2>(nullptr, nullptr, x, wq, ws, bias, N, K, y, nullptr, st)
                         : run<false, 1>(nullptr, nullptr, x, wq, ws, bias, N, K, y, nullptr, st);
  }
  if (dots) return run<true, 0>(q, s, nullptr, wq, ws, bias, N, K, y, dots, st);
  return run<false, 0>(q, s, nullptr, wq, ws, bias, N, K, y, nullptr, st);
}

}  // namespace bl
