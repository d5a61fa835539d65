// W1A8 product for large batches on the 5th-generation tensor cores
// ("binary-gemm" card, sections "API" binary_gemm and "Method"):
//   y[m,n] = bf16( s[m] * sum_k q[m,k] * w[n,k] * ws[n, k/G] + bias[n] )
// with w = +1 for a set bit, -1 for a clear one.
//
// Operands.  The MMA runs kind::f16 with fp32 accumulation.  A is the int8
// activation, exact in fp16 ((1024 + (q + 128)) - 1152).  B is the signed
// group scale +-ws[n, k/G]: the fp16 scale with its sign bit set where the
// weight bit is clear (exact).  Each product q * ws is exact in fp32 (an
// 8-bit times an 11-bit significand); the sums over K are fp32, in the
// tensor core's order (only the int32 group dots of the M <= 8 path are
// unique; here the group sums are not formed separately).
//
// Structure as the i2_s prefill kernel: one CTA per 128 x 192 output tile,
// K in blocks of 128, a 3-stage pipeline.  Warps 0-7 convert the activations
// and write them to tensor memory with tcgen05.st (the MMA reads A from
// TMEM); warps 8-15 expand the weight bits of a block into the K-major
// 128-byte-swizzled B operand in shared memory; one lane of warp 16 issues
// eight 128x192x16 MMAs per block; warps 0-15 run the epilogue (bf16 tile
// staged in shared memory, one bulk copy per row).  Every wait is bounded.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kProducers = 512;  // warps 0..15
constexpr int kThreads = 544;    // + warp 16 (TMEM, MMA issue)
constexpr int kStages = 3;
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two 64-column sub-tiles
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 256;               // activation stage st at columns 256 + 64 st
constexpr uint32_t kOutStride = BN * 2 + 16;  // staged bf16 output row, padded
constexpr uint32_t kOutBytes = BM * kOutStride;
constexpr uint32_t kPipeBytes = kStages * kBStage;
constexpr uint32_t kDataBytes = kPipeBytes > kOutBytes ? kPipeBytes : kOutBytes;
constexpr size_t kSmem = size_t(kDataBytes) + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kAcol + 64 * kStages <= kTmemCols && BN <= kAcol, "TMEM layout");

// fp32 accumulator, fp16 A and B, both K-major, N = 192, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

// byte offset of 16-byte chunk c (0..15 along K) of row r of a [rows][128]
// fp16 tile: two 64-column sub-tiles, 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  const int sub = c >> 3, cin = c & 7;
  return uint32_t(sub * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((cin ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// four int8 -> two fp16x2: (1024 + (b + 128)) - 1152 = b, exact
__device__ __forceinline__ void i8x4_to_f16(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = v ^ 0x80808080u;
  lo = hsub2(__byte_perm(x, 0x64u, 0x4140), 0x64806480u);
  hi = hsub2(__byte_perm(x, 0x64u, 0x4342), 0x64806480u);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_w1a8_tc_kernel(const int8_t* __restrict__ q, const float* __restrict__ s, const uint32_t* __restrict__ wq,
                        const uint16_t* __restrict__ ws, const uint16_t* __restrict__ bias, int M, int N, int K,
                        int G, uint16_t* __restrict__ y, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDataBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nkb = K / BK;
  const int wpr = K / 32;  // bit words per row
  const int ng = K / G;    // scale groups per row

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], kProducers);
      mbar_init(&empty[st], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 16) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp < 8) {
    // ------- activation producers: TMEM lane / tile row ra, K elements
    //         64h..64h+63 of each block (TMEM columns 32h..32h+31) -------
    const int quarter = warp & 3, h = warp >> 2;
    const int ra = quarter * 32 + lane;
    const bool a_valid = m0 + ra < M;
    const int8_t* qrow = q + int64_t(a_valid ? m0 + ra : 0) * K + 64 * h;
    const uint32_t a_taddr = tmem + (uint32_t(quarter * 32) << 16) + kAcol + 32 * h;
    auto load = [&](int kb, uint4 (&av)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        av[i] = a_valid ? *reinterpret_cast<const uint4*>(qrow + int64_t(kb) * BK + 16 * i) : make_uint4(0, 0, 0, 0);
    };
    auto produce = [&](int kb, uint4 (&av)[4]) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      tc_fence_after();
      uint4 cur[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = av[i];
      if (kb + 2 < nkb) load(kb + 2, av);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          i8x4_to_f16(cur[2 * half + i].x, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_f16(cur[2 * half + i].y, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_f16(cur[2 * half + i].z, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_f16(cur[2 * half + i].w, o[8 * i + 6], o[8 * i + 7]);
        }
        tmem_st16(a_taddr + 64 * st + 16 * half, o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[st]);
    };
    uint4 a0[4], a1[4];
    load(0, a0);
    if (nkb > 1) load(1, a1);
    for (int kb = 0; kb < nkb; kb += 2) {
      produce(kb, a0);
      if (kb + 1 < nkb) produce(kb + 1, a1);
    }
  } else if (warp < 16) {
    // ------- weight producers: 192 rows x 4 bit words (32 elements each)
    //         per block, 3 words per thread -------
    const int tb = threadIdx.x - 256;
    auto load = [&](int kb, uint32_t (&wv)[3], uint32_t (&sv)[3]) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int id = tb + 256 * i, n = id >> 2, j = id & 3;
        const bool ok = n0 + n < N;
        const int64_t row = ok ? n0 + n : 0;
        wv[i] = ok ? wq[row * wpr + kb * 4 + j] : 0u;
        const uint32_t sc = ok ? ws[row * ng + (kb * BK + 32 * j) / G] : 0u;  // rows past N: scale 0
        sv[i] = sc | (sc << 16);
      }
    };
    auto produce = [&](int kb, uint32_t (&wv)[3], uint32_t (&sv)[3]) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      uint8_t* Bs = smem + st * kBStage;
      uint32_t cw[3], cs[3];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        cw[i] = wv[i];
        cs[i] = sv[i];
      }
      if (kb + 2 < nkb) load(kb + 2, wv, sv);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int id = tb + 256 * i, n = id >> 2, j = id & 3;
        // sign bits of the 32 elements: element 2p's (inverted) bit at bit 2p'
        // of zl/zh and element 2p+1's at bit 16 + 2p' (p' = p mod 8); a left
        // shift by 15 - 2p' moves them to bits 15 and 31 of an fp16x2 word
        const uint32_t x = ~cw[i];
        const uint32_t e = x & 0x55555555u, od = (x >> 1) & 0x55555555u;
        const uint32_t zl = (e & 0xFFFFu) | (od << 16);
        const uint32_t zh = (e >> 16) | (od & 0xFFFF0000u);
#pragma unroll
        for (int step = 0; step < 4; ++step) {
          // chunk c' = (step + j) % 4 of this word (elements 8c'..8c'+7):
          // the rotation keeps each 8-thread phase on 8 distinct bank groups
          const int cq = (step + j) & 3;
          const uint32_t z = cq < 2 ? zl : zh;
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int pp = (cq & 1) * 4 + k;  // pair index within zl / zh
            o[k] = ((z << (15 - 2 * pp)) & 0x80008000u) ^ cs[i];
          }
          *reinterpret_cast<uint4*>(Bs + swz(BN, n, 4 * j + cq)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&full[st]);
    };
    uint32_t w0[3], s0[3], w1[3], s1[3];
    load(0, w0, s0);
    if (nkb > 1) load(1, w1, s1);
    for (int kb = 0; kb < nkb; kb += 2) {
      produce(kb, w0, s0);
      if (kb + 1 < nkb) produce(kb + 1, w1, s1);
    }
  } else if (lane == 0) {
    // ---------------- MMA issue (one thread) ----------------
    const uint32_t sbase = smem_addr(smem);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kStages;
      if (!*abort_flag && !mbar_wait_bounded(&full[st], uint32_t(kb / kStages) & 1u, err)) *abort_flag = 1;
      tc_fence_after();
      const uint32_t b0 = sbase + st * kBStage;
      const uint32_t a0 = tmem + kAcol + 64 * st;
      if (!*abort_flag) {
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint32_t off_b = (ks >> 2) * (BN * 128) + (ks & 3) * 32;
          umma_f16_ta(tmem, a0 + 8 * ks, umma_desc_sw128(b0 + off_b), kIdesc, (kb | ks) != 0);
        }
      }
      umma_commit(&empty[st]);
    }
    umma_commit(accum);
  }

  // ------- epilogue: warps 0-15; warp w reads TMEM lanes 32(w%4).. and
  //         columns 48(w/4) .. 48(w/4)+47 -------
  if (warp < 16) {
    if (!mbar_wait_bounded(accum, 0, err)) *abort_flag = 1;
    tc_fence_after();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int m = m0 + r;
    const int c0 = (warp >> 2) * 48;
    const float sm = (m < M) ? s[m] : 0.f;
    const bool ok = !*abort_flag;
    uint32_t v[48];
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0), *reinterpret_cast<uint32_t(*)[16]>(v));
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0 + 16), *reinterpret_cast<uint32_t(*)[16]>(v + 16));
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0 + 32), *reinterpret_cast<uint32_t(*)[16]>(v + 32));
    tmem_ld_wait();
    auto out = [&](int j) {  // bf16 bits of output column n0 + c0 + j of this row
      const int n = n0 + c0 + j;
      float b = 0.f;
      if (bias && n < N) b = bf16_bits_to_f32(bias[n]);
      return f32_to_bf16_bits_rn(__fadd_rn(__fmul_rn(__uint_as_float(v[j]), sm), b));
    };
    if ((N & 7) == 0) {
      // stage the bf16 tile in shared memory (the operand stages are free now)
      // and write each row segment with one bulk copy
      const int ncols = min(BN, N - n0);
      uint16_t* stage_row = reinterpret_cast<uint16_t*>(smem + r * kOutStride) + c0;
#pragma unroll
      for (int j = 0; j < 48; j += 8) {
        uint4 o;
        o.x = uint32_t(out(j)) | (uint32_t(out(j + 1)) << 16);
        o.y = uint32_t(out(j + 2)) | (uint32_t(out(j + 3)) << 16);
        o.z = uint32_t(out(j + 4)) | (uint32_t(out(j + 5)) << 16);
        o.w = uint32_t(out(j + 6)) | (uint32_t(out(j + 7)) << 16);
        *reinterpret_cast<uint4*>(stage_row + j) = o;
      }
      fence_async_smem();
      named_barrier_sync(1, kProducers);
      const bool issuer = threadIdx.x < BM && m0 + int(threadIdx.x) < M && ok;
      if (issuer) {
        bulk_s2g(y + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride, uint32_t(ncols) * 2);
        bulk_commit();
        bulk_wait_read();  // the global writes complete with the grid
      }
    } else if (m < M && ok) {
      for (int j = 0; j < 48; ++j) {
        const int n = n0 + c0 + j;
        if (n >= N) break;
        y[int64_t(m) * N + n] = out(j);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 16) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool w1a8_tc_applicable(int64_t M, int64_t K, int G) {
  return M > 8 && K % BK == 0 && G >= 32 && G % 32 == 0 && K % G == 0;
}

cudaError_t launch_gemm_w1a8_tc(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws,
                                const uint16_t* bias, int64_t M, int64_t N, int64_t K, int G, uint16_t* y,
                                cudaStream_t st) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = raise_smem_cap(gemm_w1a8_tc_kernel, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  return launch(gemm_w1a8_tc_kernel, grid, dim3(kThreads), kSmem, st, overlap_enabled(), q, s,
                reinterpret_cast<const uint32_t*>(wq), ws, bias, int(M), int(N), int(K), G, y, dev_error_ptr());
}

}  // namespace bl
