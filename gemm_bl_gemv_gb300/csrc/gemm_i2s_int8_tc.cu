// i2_s x int8 product on the 5th-generation tensor cores (tcgen05):
//   acc[m,n] = sum_k q[m,k] w[n,k]   (exact)
//   y[m,n]   = f32(acc[m,n]) * s[m] * scale
// ("Hesper/Layers/BitLinear", "BitLinear Mathematics", with int8 activations
// from the per-token absmax quantizer).
//
// Exactness.  The MMA runs kind::f16 (fp16 operands, fp32 accumulation).
// Activations and weights enter as power-of-two multiples of q and w whose
// products are exactly q*w (see "Scaled operands" below); every partial sum
// is an integer of magnitude <= K * 127 < 2^24 (K <= 132096), so the fp32
// accumulator holds the exact integer sum.  (This toolchain does not accept
// tcgen05 .kind::i8 for sm_103a.)
//
// Structure, one CTA per 128 x 192 output tile, K in blocks of 128 (one i2_s
// group), kStages-deep pipeline:
//   * producers read each K block from global memory two blocks ahead into
//     registers.  Warps 0-7 take the activations to tensor memory: the
//     thread of TMEM lane r converts 64 int8 of row r to fp16 and writes 32
//     columns with tcgen05.st.  Warps 8-15 expand the packed weights to fp16
//     in shared memory, in the K-major 128-byte-swizzled layout the tensor
//     core reads.  A stage is handed over with an mbarrier that all 512
//     producer threads arrive on.  Keeping the activations out of shared
//     memory halves its traffic, and separate warps let the TMEM stores
//     overlap the weight expansion.
//   * one lane of warp 16 allocates the 512 TMEM columns (accumulator
//     0..191, activation stages from 256) and issues eight 128x192x16 MMAs
//     per K block, A from TMEM, B from shared memory; tcgen05.commit frees
//     the stage and finally signals the epilogue;
//   * warps 0-15 read the accumulator (warp w: lanes 32(w%4).., 48 columns),
//     stage y in shared memory and write each row segment with one bulk
//     copy (acc likewise when asked).
// Every wait is bounded; on a timeout the CTA records the error flag,
// finishes its loops without waiting, and still frees its TMEM.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kProducers = 512;  // warps 0..15
constexpr int kThreads = 544;    // + warp 16 (TMEM, MMA issue)
constexpr int kStages = 3;
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two 64-column sub-tiles of 24 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 256;                // activation stage st at columns 256 + 64 st
constexpr uint32_t kOutStride = BN * 4 + 16;   // staged output row, padded against bank conflicts
constexpr uint32_t kOutBytes = BM * kOutStride;
constexpr uint32_t kPipeBytes = kStages * kBStage;
constexpr uint32_t kDataBytes = kPipeBytes > kOutBytes ? kPipeBytes : kOutBytes;
constexpr size_t kSmem = size_t(kDataBytes) + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kAcol + 64 * kStages <= kTmemCols && BN <= kAcol, "TMEM layout");

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both
// K-major, N = 192, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

// byte offset of 16-byte chunk `c` (0..15 along K) of row `r` inside a
// [rows][128] fp16 operand tile: two 64-column sub-tiles, 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  const int sub = c >> 3, cin = c & 7;
  return uint32_t(sub * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((cin ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// fp16 bit pattern of 2^e (-14 <= e <= 15), in both halves
__device__ __forceinline__ uint32_t f16x2_pow2(int e) {
  const uint32_t h = uint32_t(e + 15) << 10;
  return h | (h << 16);
}

// Scaled operands.  Within a 128-element group, element 32t+p of a weight
// row sits in byte p at bit 6-2t.  Masking the code in place and adding the
// fp16 exponent of 1024 gives 1024 + c*2^(6-2t); subtracting 1024 + 2^(6-2t)
// leaves 2^(6-2t) * (c - 1) = 2^(6-2t) * w (exact).  The activations of
// class t (elements 32t..32t+31) are scaled by 2^(2t-6) to match, so every
// product is exactly q*w.  Four int8 -> two fp16x2:
// ((1024 + (b + 128)) - 1152) * 2^(2t-6), one rounding of an exactly
// representable value.
__device__ __forceinline__ void i8x4_to_f16_scaled(uint32_t v, uint32_t sc, uint32_t bias, uint32_t& lo,
                                                   uint32_t& hi) {
  const uint32_t x = v ^ 0x80808080u;
  lo = hfma2(__byte_perm(x, 0x64u, 0x4140), sc, bias);
  hi = hfma2(__byte_perm(x, 0x64u, 0x4342), sc, bias);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_i2s_int8_tc_kernel(const int8_t* __restrict__ q, const float* __restrict__ s,
                            const uint8_t* __restrict__ packed, int M, int N, int K, float* __restrict__ y,
                            int32_t* __restrict__ acc_out, unsigned int* err) {
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
  const int64_t row_bytes = K / 4;

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
  pdl_wait();

  if (warp < 8) {
    // ------- activation producers: the thread owns TMEM lane / tile row ra
    //         and K elements 64h..64h+63 of each block (classes 2h, 2h+1;
    //         TMEM columns 32h..32h+31 of the stage) -------
    const int quarter = warp & 3, h = warp >> 2;
    const int ra = quarter * 32 + lane;
    const bool a_valid = m0 + ra < M;
    const int8_t* qrow = q + int64_t(a_valid ? m0 + ra : 0) * K + 64 * h;
    const uint32_t sc0 = f16x2_pow2(4 * h - 6), sc1 = f16x2_pow2(4 * h - 4);
    const uint32_t bias0 = hfma2(0x64806480u, sc0, 0x80008000u) ^ 0x80008000u;  // -(1152 * scale)
    const uint32_t bias1 = hfma2(0x64806480u, sc1, 0x80008000u) ^ 0x80008000u;
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
        const uint32_t sc = half ? sc1 : sc0, bias = half ? bias1 : bias0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          i8x4_to_f16_scaled(cur[2 * half + i].x, sc, bias, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_f16_scaled(cur[2 * half + i].y, sc, bias, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_f16_scaled(cur[2 * half + i].z, sc, bias, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_f16_scaled(cur[2 * half + i].w, sc, bias, o[8 * i + 6], o[8 * i + 7]);
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
    // ------- weight producers: 192 rows x 4 pieces of 8 bytes, 3 per thread -------
    const int tb = threadIdx.x - 256;
    auto load = [&](int kb, uint2 (&bv)[3]) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int id = tb + 256 * i, n = id >> 2, j = id & 3;
        bv[i] = (n0 + n < N) ? *reinterpret_cast<const uint2*>(packed + int64_t(n0 + n) * row_bytes + 32 * kb + 8 * j)
                             : make_uint2(0x55555555u, 0x55555555u);  // code 01 = weight 0
      }
    };
    auto produce = [&](int kb, uint2 (&bv)[3]) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      uint8_t* Bs = smem + st * kBStage;
      uint2 cur[3];
#pragma unroll
      for (int i = 0; i < 3; ++i) cur[i] = bv[i];
      if (kb + 2 < nkb) load(kb + 2, bv);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int id = tb + 256 * i, n = id >> 2, j = id & 3;
        // bytes 8j..8j+7 of the group, spread so byte p lands in an fp16 half
        const uint32_t pr[4] = {__byte_perm(cur[i].x, 0u, 0x4140), __byte_perm(cur[i].x, 0u, 0x4342),
                                __byte_perm(cur[i].y, 0u, 0x4140), __byte_perm(cur[i].y, 0u, 0x4342)};
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          // odd rows visit the classes as 1,0,3,2 so an 8-thread phase (two
          // rows) covers all 8 bank groups
          const int t = tt ^ (n & 1);
          const uint32_t mask = 0x00030003u << (6 - 2 * t);
          const uint32_t off = 0x64006400u | (0x00010001u << (6 - 2 * t));  // 1024 + 2^(6-2t)
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = hsub2((pr[k] & mask) | 0x64006400u, off);
          *reinterpret_cast<uint4*>(Bs + swz(BN, n, 4 * t + j)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&full[st]);
    };
    uint2 b0[3], b1[3];
    load(0, b0);
    if (nkb > 1) load(1, b1);
    for (int kb = 0; kb < nkb; kb += 2) {
      produce(kb, b0);
      if (kb + 1 < nkb) produce(kb + 1, b1);
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

  // ------- epilogue: warps 0-15; warp w reads TMEM lanes 32(w%4).. (its rows)
  //         and columns 48(w/4) .. 48(w/4)+47 -------
  if (warp < 16) {
    if (!mbar_wait_bounded(accum, 0, err)) *abort_flag = 1;
    tc_fence_after();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int m = m0 + r;
    const int c0 = (warp >> 2) * 48;
    const float sm = (m < M) ? s[m] : 0.f;
    const float sw = *reinterpret_cast<const float*>(packed + int64_t(N) * row_bytes);
    const bool ok = !*abort_flag;
    uint32_t v[48];
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0), *reinterpret_cast<uint32_t(*)[16]>(v));
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0 + 16), *reinterpret_cast<uint32_t(*)[16]>(v + 16));
    tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0 + 32), *reinterpret_cast<uint32_t(*)[16]>(v + 32));
    tmem_ld_wait();
    if ((N & 3) == 0) {
      // stage the tile in shared memory (the operand stages are free now) and
      // write each row segment with one bulk copy
      const int ncols = min(BN, N - n0);
      float* stage_row = reinterpret_cast<float*>(smem + r * kOutStride) + c0;
#pragma unroll
      for (int j = 0; j < 48; j += 4) {
        float4 o;
        o.x = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
        o.y = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 1]), sm), sw);
        o.z = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 2]), sm), sw);
        o.w = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 3]), sm), sw);
        *reinterpret_cast<float4*>(stage_row + j) = o;
      }
      fence_async_smem();
      named_barrier_sync(1, kProducers);
      const bool issuer = threadIdx.x < BM && m0 + int(threadIdx.x) < M && ok;
      if (issuer) {
        bulk_s2g(y + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride, uint32_t(ncols) * 4);
        bulk_commit();
      }
      if (acc_out) {
        if (issuer) bulk_wait_read();
        named_barrier_sync(1, kProducers);
        int* stage_acc = reinterpret_cast<int*>(smem + r * kOutStride) + c0;
#pragma unroll
        for (int j = 0; j < 48; j += 4)
          *reinterpret_cast<int4*>(stage_acc + j) =
              make_int4(__float2int_rn(__uint_as_float(v[j])), __float2int_rn(__uint_as_float(v[j + 1])),
                        __float2int_rn(__uint_as_float(v[j + 2])), __float2int_rn(__uint_as_float(v[j + 3])));
        fence_async_smem();
        named_barrier_sync(1, kProducers);
        if (issuer) {
          bulk_s2g(acc_out + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride,
                   uint32_t(ncols) * 4);
          bulk_commit();
        }
      }
      if (issuer) bulk_wait();
    } else if (m < M && ok) {
      for (int j = 0; j < 48; ++j) {
        const int n = n0 + c0 + j;
        if (n >= N) break;
        y[int64_t(m) * N + n] = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
        if (acc_out) acc_out[int64_t(m) * N + n] = __float2int_rn(__uint_as_float(v[j]));
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
  pdl_launch_dependents();
}

}  // namespace

// Tensor-core path: M >= 64 (smaller batches use the CUDA-core kernel).
cudaError_t launch_gemm_i2s_int8(const int8_t* q, const float* sc, const uint8_t* packed, int64_t M, int64_t N,
                                 int64_t K, float* y, int32_t* acc, cudaStream_t s) {
  if (M < 64) return launch_gemm_i2s_int8_simt(q, sc, packed, M, N, K, y, acc, s);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = raise_smem_cap(gemm_i2s_int8_tc_kernel, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  return launch(gemm_i2s_int8_tc_kernel, grid, dim3(kThreads), kSmem, s, overlap_enabled(), q, sc, packed, int(M),
                int(N), int(K), y, acc, dev_error_ptr());
}

}  // namespace bl
