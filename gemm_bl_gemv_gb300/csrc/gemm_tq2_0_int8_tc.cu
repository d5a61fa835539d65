// TQ2_0 weights against int8 activations, large batches, on the
// 5th-generation tensor cores ("Hesper/Quantization/TQ2_0", "TQ2_0 Format",
// with the activations of the "binary-gemm" card's quantize_activation):
//   y[m,n] = s[m] * sum_k q[m,k] * w[n,k] * d[n, k/256]          (fp32)
//
// Operands.  The MMA runs kind::f16 with fp32 accumulation.  Element k of a
// K block carries the power of two S = 4^(k % 4) on the weight side and 1/S
// on the activation side: A = q / S and B = w * d * S, both exact in fp16
// (q has 8 significant bits; w * d * S is d times a power of two up to 64,
// exact while |d| < 1024, subnormal d included).  Every product is then
// exactly q * w * d in fp32 and the sum over K is fp32 in the tensor core's
// order.
//
// B decode.  A TQ2_0 code is the 2-bit two's complement of w (00 -> 0,
// 01 -> +1, 11 -> -1), so XOR with 10b gives the offset form f = w + 2.  The
// 8 codes of a 16-bit word, copied into both halves of a register, already
// sit where the S above puts them: element e's field at bit 2(e % 4) of the
// half (elements 4..7 after one shift by 8), i.e. f * S in the mantissa.  One
// LOP3 keeps a pair's two fields, flips them to f and sets the fp16 exponent
// of 1024 (1024 + f S per half); one f16x2 subtraction of 1024 + 2 S leaves
// w S exactly and one f16x2 multiply by (d, d) gives the operand pair.  The
// activation conversion folds 1/S into its f16x2 FMA.
//
// Loads.  The activation tile of a K block (128 tokens x 128 bytes) arrives
// by one TMA load with the 128-byte swizzle.  TQ2_0 blocks are 66 bytes, so
// weight rows are only 2-byte aligned: each decoding lane loads one 16-bit
// word (8 codes, one 16-byte operand chunk) and 16 lanes cover the 32 code
// bytes of a row, two rows per warp load.  A 128-element K block is half a
// TQ2_0 block.
//
// Structure: one CTA per 128 x 192 output tile, K in blocks of 128, a
// 3-stage pipeline.  Warps 0-3 convert the activations and write them to
// tensor memory with tcgen05.st (the MMA reads A from TMEM); warps 4-19
// decode the weights into the K-major 128-byte-swizzled B operand in shared
// memory; one lane of warp 20 issues eight 128x192x16 MMAs per block; warp 21
// issues the activation TMA loads; warps 0-15 run the epilogue (fp32 tile
// staged in shared memory, one bulk copy per row).  Every wait is bounded.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kAWarps = 4;                    // activation warps, one per TMEM lane quarter
constexpr int kBWarps = 16;                   // weight decoding warps
constexpr int kProducers = 32 * (kAWarps + kBWarps);
constexpr int kBThreads = 32 * kBWarps;
constexpr int kChunks = BN * (BK / 8) / kBThreads;  // 16-byte B chunks per decoding thread and block
static_assert(kChunks * kBThreads == BN * (BK / 8), "chunks must divide evenly");
constexpr int kMmaWarp = kAWarps + kBWarps;   // TMEM allocation, MMA issue
constexpr int kThreads = 32 * (kMmaWarp + 2);  // + one warp of activation TMA loads
constexpr int kEpilogue = 512;                // warps 0..15 run the epilogue
constexpr int kStages = 3;
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two 64-column sub-tiles
constexpr uint32_t kAStage = BM * BK;      // 16 KB of int8 activations, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 256;               // activation stage st at columns 256 + 64 st
constexpr uint32_t kOutStride = BN * 4 + 16;  // staged fp32 output row, padded
constexpr uint32_t kOutBytes = BM * kOutStride;
constexpr uint32_t kPipeBytes = kStages * kBStage;
constexpr uint32_t kDataBytes = kPipeBytes > kOutBytes ? kPipeBytes : kOutBytes;
constexpr uint32_t kAOff = kDataBytes;  // 1024-aligned (the swizzle repeats every 1024 bytes)
constexpr uint32_t kBarOff = kAOff + kStages * kAStage;
constexpr size_t kSmem = size_t(kBarOff) + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kAcol + 64 * kStages <= kTmemCols && BN <= kAcol, "TMEM layout");
static_assert(kAOff % 1024 == 0, "swizzled TMA destination");

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

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// four int8 (elements 4m .. 4m+3) -> two fp16x2 of q / S, S = 1, 4, 16, 64:
// (1152 + q) / S - 1152 / S = q / S, one rounding of an exact value
__device__ __forceinline__ void i8x4_to_f16_scaled(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = v ^ 0x80808080u;
  lo = hfma2(__byte_perm(x, 0x64u, 0x4140), 0x34003C00u /* 1/4, 1 */, 0xDC80E480u /* -288, -1152 */);
  hi = hfma2(__byte_perm(x, 0x64u, 0x4342), 0x24002C00u /* 1/64, 1/16 */, 0xCC80D480u /* -18, -72 */);
}

// The 8 codes of one 16-bit word (element e at bits 2e, 2e+1) -> four fp16x2
// words of w * d * S, elements (2k, 2k+1) in word k; ds = (d, d).
__device__ __forceinline__ uint4 tq2_chunk(uint32_t c, uint32_t ds) {
  const uint32_t w = c * 0x00010001u;  // the codes in both halves
  const uint32_t w8 = w >> 8;          // elements 4..7 in the low bytes of both halves
  // (w & M) ^ K: the two fields of a pair, flipped to f, under the exponent of 1024
  const uint32_t p0 = (w & 0x000C0003u) ^ 0x64086402u, p1 = (w & 0x00C00030u) ^ 0x64806420u;
  const uint32_t p2 = (w8 & 0x000C0003u) ^ 0x64086402u, p3 = (w8 & 0x00C00030u) ^ 0x64806420u;
  // minus (1024 + 2 S): w S exactly; times (d, d)
  return make_uint4(hmul2(hsub2(p0, 0x64086402u), ds), hmul2(hsub2(p1, 0x64806420u), ds),
                    hmul2(hsub2(p2, 0x64086402u), ds), hmul2(hsub2(p3, 0x64806420u), ds));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tq2_0_int8_tc_kernel(const __grid_constant__ CUtensorMap qmap, const float* __restrict__ s,
                              const uint8_t* __restrict__ packed, int M, int N, int K, float* __restrict__ y,
                              unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* araw = smem + kAOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* a_full = empty + kStages;
  uint64_t* a_empty = a_full + kStages;
  uint64_t* accum = a_empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nkb = K / BK;
  const int64_t nb = K / 256;  // TQ2_0 blocks per row

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], kProducers);
      mbar_init(&empty[st], 1);
      mbar_init(&a_full[st], 1);
      mbar_init(&a_empty[st], 32 * kAWarps);
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
      if (!*abort_flag && !mbar_wait_bounded(&a_full[st], uint32_t(kb / kStages) & 1u, err)) *abort_flag = 1;
      tc_fence_after();
      // row ra of the swizzled tile: chunk c at 16 * (c ^ (ra % 8))
      const uint8_t* arow = araw + st * kAStage + ra * 128;
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = *reinterpret_cast<const uint4*>(arow + ((c ^ (ra & 7)) << 4));
      mbar_arrive(&a_empty[st]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {  // chunks 2h, 2h+1 -> TMEM columns 16h..16h+15
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 c = v[2 * h + i];
          i8x4_to_f16_scaled(c.x, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_f16_scaled(c.y, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_f16_scaled(c.z, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_f16_scaled(c.w, o[8 * i + 6], o[8 * i + 7]);
        }
        tmem_st16(a_taddr + 64 * st + 16 * h, o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[st]);
    }
  } else if (warp < kMmaWarp) {
    // ------- weight decoders: chunk g = tb + kBThreads i of a block is
    //         row g / 16, elements 8 (g % 16) .. 8 (g % 16) + 7 -------
    const int tb = threadIdx.x - 32 * kAWarps;
    const int cofs = 2 * (tb & 15);  // kBThreads is a multiple of 16: g % 16 = tb % 16 for every chunk
    const uint8_t* rowp[kChunks];    // row start + 2 (g % 16)
    uint32_t sto[kChunks];         // byte offset of the chunk in a stage
    uint32_t valid = 0;            // bit i: the chunk's row is below N
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int g = tb + kBThreads * i, n = g >> 4, c = g & 15;
      const bool ok = n0 + n < N;
      valid |= uint32_t(ok) << i;
      rowp[i] = packed + (ok ? int64_t(n0 + n) * nb * 66 : 0) + 2 * c;
      sto[i] = uint32_t((c >> 3) * (BN * 128) + (n >> 3) * 1024 + (n & 7) * 128 + (((c & 7) ^ (n & 7)) << 4));
    }
    uint32_t dmax = 0;  // largest |d| bit pattern seen
    auto load = [&](int kb, uint32_t (&cv)[kChunks], uint32_t (&dv)[kChunks]) {
      const int off = 66 * (kb >> 1) + 32 * (kb & 1);  // codes of K block kb
      const int doff = 66 * (kb >> 1) + 64;            // the block scale
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        cv[i] = dv[i] = 0u;  // rows past N: zero operand
        if ((valid >> i) & 1u) {
          cv[i] = __ldg(reinterpret_cast<const uint16_t*>(rowp[i] + off));
          dv[i] = __ldg(reinterpret_cast<const uint16_t*>(rowp[i] + doff - cofs));
        }
      }
    };
    auto produce = [&](int kb, uint32_t (&cv)[kChunks], uint32_t (&dv)[kChunks]) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      uint8_t* Bs = smem + st * kBStage;
      uint32_t cur[kChunks], dcur[kChunks];
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        cur[i] = cv[i];
        dcur[i] = dv[i];
      }
      if (kb + 2 < nkb) load(kb + 2, cv, dv);
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        if ((kb & 1) == 0) dmax = max(dmax, dcur[i] & 0x7FFFu);  // once per TQ2_0 block
        *reinterpret_cast<uint4*>(Bs + sto[i]) = tq2_chunk(cur[i], dcur[i] * 0x00010001u);
      }
      fence_async_smem();
      mbar_arrive(&full[st]);
    };
    uint32_t c0[kChunks], d0[kChunks], c1[kChunks], d1[kChunks];
    load(0, c0, d0);
    if (nkb > 1) load(1, c1, d1);
    for (int kb = 0; kb < nkb; kb += 2) {
      produce(kb, c0, d0);
      if (kb + 1 < nkb) produce(kb + 1, c1, d1);
    }
    if (dmax >= 0x6400u && err) atomicOr(err, BL_DEVERR_RANGE);  // |d| >= 1024: w d S may overflow fp16
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
    // ---------------- activation TMA loads (one thread) ----------------
    int issued = 0;
    for (int kb = 0; kb < nkb && !*abort_flag; ++kb) {
      const int st = kb % kStages;
      if (kb >= kStages && !mbar_wait_bounded(&a_empty[st], uint32_t(kb / kStages - 1) & 1u, err)) {
        *abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(&a_full[st], kAStage);
      tma_load_2d(araw + st * kAStage, &qmap, kb * BK, m0, &a_full[st]);
      issued = kb + 1;
    }
    // the CTA must not finish while a load still writes its shared memory
    for (int kb = issued - kStages < 0 ? 0 : issued - kStages; kb < issued; ++kb)
      mbar_wait_bounded(&a_full[kb % kStages], uint32_t(kb / kStages) & 1u, nullptr);
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
    if ((N & 3) == 0) {
      // stage the fp32 tile in shared memory (the operand stages are free now)
      // and write each row segment with one bulk copy
      const int ncols = min(BN, N - n0);
      float* stage_row = reinterpret_cast<float*>(smem + r * kOutStride) + c0;
#pragma unroll
      for (int j = 0; j < 48; j += 4) {
        float4 o;
        o.x = __fmul_rn(__uint_as_float(v[j]), sm);
        o.y = __fmul_rn(__uint_as_float(v[j + 1]), sm);
        o.z = __fmul_rn(__uint_as_float(v[j + 2]), sm);
        o.w = __fmul_rn(__uint_as_float(v[j + 3]), sm);
        *reinterpret_cast<float4*>(stage_row + j) = o;
      }
      fence_async_smem();
      named_barrier_sync(1, kEpilogue);
      const bool issuer = threadIdx.x < BM && m0 + int(threadIdx.x) < M && ok;
      if (issuer) {
        bulk_s2g(y + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride, uint32_t(ncols) * 4);
        bulk_commit();
        bulk_wait_read();  // the global writes complete with the grid
      }
    } else if (m < M && ok) {
      for (int j = 0; j < 48; ++j) {
        const int n = n0 + c0 + j;
        if (n >= N) break;
        y[int64_t(m) * N + n] = __fmul_rn(__uint_as_float(v[j]), sm);
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

cudaError_t launch_gemm_tq2_0_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N,
                                   int64_t K, float* y, cudaStream_t st) {
  int dev = 0;
  cudaGetDevice(&dev);
  CUtensorMap qmap;  // q as [M][K] bytes, boxes of 128 tokens x 128 bytes
  if (!encode_tmap_2d_u8(&qmap, q, uint64_t(K), uint64_t(M), uint64_t(K), BK, BM, true)) return cudaErrorNotSupported;
  cudaError_t e = raise_smem_cap(gemm_tq2_0_int8_tc_kernel, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  return launch(gemm_tq2_0_int8_tc_kernel, grid, dim3(kThreads), kSmem, st, overlap_enabled(), qmap, s, packed,
                int(M), int(N), int(K), y, dev_error_ptr());
}

}  // namespace bl
