// W1A8 product for large batches on the 5th-generation tensor cores
// ("binary-gemm" card, sections "API" binary_gemm and "Method"):
//   y[m,n] = bf16( s[m] * sum_k q[m,k] * w[n,k] * ws[n, k/G] + bias[n] )
// with w = +1 for a set bit, -1 for a clear one.
//
// Operands.  The MMA runs kind::f16 with fp32 accumulation.  A is the int8
// activation, exact in fp16 ((1024 + (q + 128)) - 1152).  B is the signed
// group scale +-ws[n, k/G]: the fp16 scale with its sign bit flipped where
// the weight bit is clear (exact).  Each product q * ws is exact in fp32 (an
// 8-bit times an 11-bit significand); the sums over K are fp32, in the
// tensor core's order (only the int32 group dots of the M <= 8 path are
// unique; here the group sums are not formed separately).
//
// B decode.  Byte b of a bit word holds elements 8c..8c+7.  Multiplying b by
// 2^(15-2k) + 2^(30-2k) puts bit 2k at bit 15 and bit 2k+1 at bit 31 (the two
// shifted copies never overlap), so one LOP3 of the inverted product with
// 0x80008000 and the scale pair (ws, ws) gives the fp16x2 word of elements
// 2k, 2k+1: one byte select, four IMAD and four LOP3 per 8 weights.
//
// Structure as the i2_s prefill kernel: one CTA per 128 x 192 output tile,
// K in blocks of 128, a 3-stage pipeline.  Warp 17 brings each K block's
// 128 x 128 activation tile (128-byte swizzle) and 192 x 16 bytes of bit
// words with two TMA loads; warps 0-3 convert the activations and write them
// to tensor memory with tcgen05.st (the MMA reads A from TMEM); warps 4-15
// build the B operand in shared memory (K-major, 128-byte swizzle; the group
// scales are read from global memory two blocks ahead); one lane of warp 16
// issues eight 128x192x16 MMAs per block; warps 0-15 run the epilogue (bf16
// tile staged in shared memory, one bulk copy per row).  Every wait is
// bounded.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kAWarps = 4;                    // activation warps, one per TMEM lane quarter
constexpr int kBWarps = 12;                   // B operand warps
constexpr int kProducers = 32 * (kAWarps + kBWarps);
constexpr int kBThreads = 32 * kBWarps;
constexpr int kRuns = BN * 4 / kBThreads;     // 32-bit words (32 elements) per B thread and block
static_assert(kRuns * kBThreads == BN * 4 && (kBWarps * kRuns) % 24 == 0, "runs must divide evenly");
constexpr int kMmaWarp = kAWarps + kBWarps;   // TMEM allocation, MMA issue
constexpr int kThreads = 32 * (kMmaWarp + 2);  // + one warp of TMA loads
constexpr int kEpilogue = 512;                // warps 0..15 run the epilogue
constexpr int kStages = 3;
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two 64-column sub-tiles
constexpr uint32_t kAStage = BM * BK;      // 16 KB of int8 activations, 128-byte swizzled
constexpr uint32_t kWStage = BN * BK / 8;  // 3 KB of bit words, 16 bytes per row
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 256;               // activation stage st at columns 256 + 64 st
constexpr uint32_t kOutStride = BN * 2 + 16;  // staged bf16 output row, padded
constexpr uint32_t kOutBytes = BM * kOutStride;
constexpr uint32_t kPipeBytes = kStages * kBStage;
constexpr uint32_t kDataBytes = kPipeBytes > kOutBytes ? kPipeBytes : kOutBytes;
constexpr uint32_t kAOff = kDataBytes;  // 1024-aligned (the swizzle repeats every 1024 bytes)
constexpr uint32_t kWOff = kAOff + kStages * kAStage;
constexpr uint32_t kBarOff = kWOff + kStages * kWStage;
constexpr size_t kSmem = size_t(kBarOff) + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kAcol + 64 * kStages <= kTmemCols && BN <= kAcol, "TMEM layout");
static_assert(kAOff % 1024 == 0 && kWOff % 128 == 0 && kWStage % 128 == 0, "TMA destinations");

// fp32 accumulator, fp16 A and B, both K-major, N = 192, M = 128.  The B
// stage is [192 rows][128 K] fp16 as two 64-column sub-tiles, 128-byte
// swizzled: 16-byte chunk c of row n sits at
//   (c / 8) * 192 * 128 + (n / 8) * 1024 + (n % 8) * 128 + ((c % 8) ^ (n % 8)) * 16.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

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

// byte b of weight bits (element e at bit e) and the scale pair cs = (ws, ws)
// -> four fp16x2 words of +-ws, elements (2k, 2k+1) in word k
__device__ __forceinline__ uint4 w1_chunk(uint32_t b, uint32_t cs) {
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t x = b * ((1u << (15 - 2 * k)) + (1u << (30 - 2 * k)));  // bits 2k, 2k+1 -> 15, 31
    o[k] = (~x & 0x80008000u) ^ cs;                                           // sign set where the bit is clear
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_w1a8_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                        const float* __restrict__ s, const uint16_t* __restrict__ ws,
                        const uint16_t* __restrict__ bias, int M, int N, int K, int G, uint16_t* __restrict__ y,
                        unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* araw = smem + kAOff;
  uint8_t* wraw = smem + kWOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* raw_full = empty + kStages;
  uint64_t* raw_empty = raw_full + kStages;
  uint64_t* accum = raw_empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nkb = K / BK;
  const int ng = K / G;  // scale groups per row

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], kProducers);
      mbar_init(&empty[st], 1);
      mbar_init(&raw_full[st], 1);
      mbar_init(&raw_empty[st], kProducers);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp < kAWarps) {
    // ------- activation converters: TMEM lane / tile row ra, all 128 K
    //         elements of a block (TMEM columns 0..63 of the stage) -------
    const int ra = warp * 32 + lane;
    const uint32_t a_taddr = tmem + (uint32_t(warp * 32) << 16) + kAcol;
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      if (!*abort_flag && !mbar_wait_bounded(&raw_full[st], uint32_t(kb / kStages) & 1u, err)) *abort_flag = 1;
      tc_fence_after();
      // row ra of the swizzled tile: chunk c at 16 * (c ^ (ra % 8))
      const uint8_t* arow = araw + st * kAStage + ra * 128;
#pragma unroll
      for (int h = 0; h < 4; ++h) {  // chunks 2h, 2h+1 -> TMEM columns 16h..16h+15
        uint4 v[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) v[i] = *reinterpret_cast<const uint4*>(arow + (((2 * h + i) ^ (ra & 7)) << 4));
        if (h == 3) mbar_arrive(&raw_empty[st]);
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          i8x4_to_f16(v[i].x, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_f16(v[i].y, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_f16(v[i].z, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_f16(v[i].w, o[8 * i + 6], o[8 * i + 7]);
        }
        tmem_st16(a_taddr + 64 * st + 16 * h, o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[st]);
    }
  } else if (warp < kMmaWarp) {
    // ------- B operand: run i of a thread is row n = 8 R + lane % 8
    //         (R = B warp + kBWarps i) and bit word j = lane / 8 of the
    //         block (elements 32j..32j+31, 16-byte chunks 4j..4j+3) -------
    const int wb = warp - kAWarps;
    const int r = lane & 7, j = lane >> 3;
    const uint32_t u = uint32_t((4 * (j & 1)) ^ r);  // chunk 4j + c lands in 16-byte unit u ^ c, sub-tile j / 2
    uint32_t rofs[kRuns], sto[kRuns];
    const uint16_t* srow[kRuns];
    bool valid[kRuns];
#pragma unroll
    for (int i = 0; i < kRuns; ++i) {
      const int R = wb + kBWarps * i, n = 8 * R + r;
      valid[i] = n0 + n < N;
      srow[i] = ws + (valid[i] ? int64_t(n0 + n) * ng : 0);
      rofs[i] = uint32_t(n * 16 + 4 * j);
      sto[i] = uint32_t((j >> 1) * (BN * 128) + R * 1024 + r * 128);
    }
    // the group scales of block kb, in both halves (rows past N: 0)
    auto load = [&](int kb, uint32_t (&sv)[kRuns]) {
      const int g = (kb * BK + 32 * j) / G;
#pragma unroll
      for (int i = 0; i < kRuns; ++i) sv[i] = valid[i] ? uint32_t(srow[i][g]) * 0x00010001u : 0u;
    };
    auto produce = [&](int kb, uint32_t (&sv)[kRuns]) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      if (!*abort_flag && !mbar_wait_bounded(&raw_full[st], uint32_t(kb / kStages) & 1u, err)) *abort_flag = 1;
      uint32_t wd[kRuns], cs[kRuns];
#pragma unroll
      for (int i = 0; i < kRuns; ++i) {
        wd[i] = *reinterpret_cast<const uint32_t*>(wraw + st * kWStage + rofs[i]);
        cs[i] = sv[i];
      }
      mbar_arrive(&raw_empty[st]);
      if (kb + 2 < nkb) load(kb + 2, sv);
      uint8_t* Bs = smem + st * kBStage;
#pragma unroll
      for (int i = 0; i < kRuns; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(Bs + sto[i] + ((u ^ uint32_t(c)) << 4)) =
              w1_chunk(__byte_perm(wd[i], 0u, 0x4440u + uint32_t(c)), cs[i]);
      fence_async_smem();
      mbar_arrive(&full[st]);
    };
    uint32_t s0[kRuns], s1[kRuns];
    load(0, s0);
    if (nkb > 1) load(1, s1);
    for (int kb = 0; kb < nkb; kb += 2) {
      produce(kb, s0);
      if (kb + 1 < nkb) produce(kb + 1, s1);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
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
  } else if (lane == 0) {
    // ---------------- TMA loads of the raw operands (one thread) ----------------
    int issued = 0;
    for (int kb = 0; kb < nkb && !*abort_flag; ++kb) {
      const int st = kb % kStages;
      if (kb >= kStages && !mbar_wait_bounded(&raw_empty[st], uint32_t(kb / kStages - 1) & 1u, err)) {
        *abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(&raw_full[st], kAStage + kWStage);
      tma_load_2d(araw + st * kAStage, &qmap, kb * BK, m0, &raw_full[st]);
      tma_load_2d(wraw + st * kWStage, &wmap, kb * (BK / 8), n0, &raw_full[st]);
      issued = kb + 1;
    }
    // the CTA must not finish while a load still writes its shared memory
    for (int kb = issued - kStages < 0 ? 0 : issued - kStages; kb < issued; ++kb)
      mbar_wait_bounded(&raw_full[kb % kStages], uint32_t(kb / kStages) & 1u, nullptr);
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
      named_barrier_sync(1, kEpilogue);
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
  if (warp == kMmaWarp) {
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
  CUtensorMap qmap, wmap;  // q as [M][K] bytes (128 x 128 boxes, swizzled); bits as [N][K/8] bytes (192 x 16)
  if (!encode_tmap_2d_u8(&qmap, q, uint64_t(K), uint64_t(M), uint64_t(K), BK, BM, true) ||
      !encode_tmap_2d_u8(&wmap, wq, uint64_t(K / 8), uint64_t(N), uint64_t(K / 8), BK / 8, BN, false))
    return cudaErrorNotSupported;
  cudaError_t e = raise_smem_cap(gemm_w1a8_tc_kernel, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  return launch(gemm_w1a8_tc_kernel, grid, dim3(kThreads), kSmem, st, overlap_enabled(), qmap, wmap, s, ws, bias,
                int(M), int(N), int(K), G, y, dev_error_ptr());
}

}  // namespace bl
