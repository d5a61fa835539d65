// i2_s x int8 product on the 5th-generation tensor cores (tcgen05):
//   acc[m,n] = sum_k q[m,k] w[n,k]   (exact)
//   y[m,n]   = f32(acc[m,n]) * s[m] * scale
// ("Hesper/Layers/BitLinear", "BitLinear Mathematics", with int8 activations
// from the per-token absmax quantizer).
//
// Exactness.  The MMA runs kind::f16 (fp16 operands, fp32 accumulation): an
// int8 activation and a ternary weight are exact in fp16, their product is
// exact, and every partial sum is an integer of magnitude <= K * 127 < 2^24
// (K <= 132096), so the fp32 accumulator holds the exact integer sum.  (This
// toolchain does not accept tcgen05 .kind::i8 for sm_103a.)
//
// Structure, one CTA per 128 x 192 output tile, K in blocks of 128 (one i2_s
// group):
//   * warps 0-7 (producers) read the activation rows (int8) and the packed
//     weight rows for a K block from global memory, convert them to fp16
//     (activations with the 1024+u magic-number trick, ternary codes the same
//     way) and write both operands into a shared-memory stage in the K-major
//     128-byte-swizzled layout the tensor core reads; a stage is handed over
//     with an mbarrier;
//   * one lane of warp 8 allocates 256 TMEM columns and issues eight
//     128x192x16 MMAs per K block; tcgen05.commit releases the stage when
//     they complete and, after the last block, signals the epilogue;
//   * warps 0-3 read the accumulator from TMEM (each warp its 32 lanes = 32
//     rows) and write y (and acc when asked).
// Every wait is bounded; on a timeout the CTA records the error flag,
// finishes its loops without waiting, and still frees its TMEM.
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kProducers = 256;  // warps 0..7
constexpr int kThreads = 288;    // + warp 8 (TMEM, MMA issue)
constexpr int kStages = 2;
constexpr uint32_t kAStage = BM * BK * 2;  // 32 KB: two 64-column sub-tiles of 16 KB
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two sub-tiles of 24 KB
constexpr uint32_t kStageBytes = kAStage + kBStage;
constexpr uint32_t kTmemCols = 256;
constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

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

// four int8 -> two fp16x2: (1024 + (b + 128)) - 1152 = b, exact
__device__ __forceinline__ void i8x4_to_f16(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = v ^ 0x80808080u;
  lo = hsub2(__byte_perm(x, 0x64u, 0x4140), 0x64806480u);
  hi = hsub2(__byte_perm(x, 0x64u, 0x4342), 0x64806480u);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_i2s_int8_tc_kernel(const int8_t* __restrict__ q, const float* __restrict__ s,
                            const uint8_t* __restrict__ packed, int M, int N, int K, float* __restrict__ y,
                            int32_t* __restrict__ acc_out, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
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
  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp < 8) {
    // ---------------- producers ----------------
    const int tid = threadIdx.x;
    uint4 av[4];
    uint2 bv[3];
    auto load = [&](int kb) {
      const int k0 = kb * BK;
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // activations: 128 rows x 8 chunks of 16 bytes
        const int id = tid + kProducers * i, r = id >> 3, j = id & 7;
        av[i] = (m0 + r < M) ? *reinterpret_cast<const uint4*>(q + int64_t(m0 + r) * K + k0 + 16 * j)
                             : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 3; ++i) {  // weights: 192 rows x 4 pieces of 8 bytes (one 32-byte group)
        const int id = tid + kProducers * i, n = id >> 2, j = id & 3;
        bv[i] = (n0 + n < N) ? *reinterpret_cast<const uint2*>(packed + int64_t(n0 + n) * row_bytes + 32 * kb + 8 * j)
                             : make_uint2(0x55555555u, 0x55555555u);  // code 01 = weight 0
      }
    };
    load(0);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb & 1;
      if (kb >= kStages && !*abort_flag && !mbar_wait_bounded(&empty[st], uint32_t((kb >> 1) - 1) & 1u, err))
        *abort_flag = 1;
      uint8_t* As = smem + st * kStageBytes;
      uint8_t* Bs = As + kAStage;
      const uint4 a_cur[4] = {av[0], av[1], av[2], av[3]};
      const uint2 b_cur[3] = {bv[0], bv[1], bv[2]};
      if (kb + 1 < nkb) load(kb + 1);  // prefetch the next block while converting this one
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int id = tid + kProducers * i, r = id >> 3, j = id & 7;
        uint4 o0, o1;
        i8x4_to_f16(a_cur[i].x, o0.x, o0.y);
        i8x4_to_f16(a_cur[i].y, o0.z, o0.w);
        i8x4_to_f16(a_cur[i].z, o1.x, o1.y);
        i8x4_to_f16(a_cur[i].w, o1.z, o1.w);
        *reinterpret_cast<uint4*>(As + swz(BM, r, 2 * j)) = o0;
        *reinterpret_cast<uint4*>(As + swz(BM, r, 2 * j + 1)) = o1;
      }
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int id = tid + kProducers * i, n = id >> 2, j = id & 3;
        // bytes 8j..8j+7 of the group; element 32t+p sits in byte p at shift 6-2t
        const uint32_t pr[4] = {__byte_perm(b_cur[i].x, 0u, 0x4140), __byte_perm(b_cur[i].x, 0u, 0x4342),
                                __byte_perm(b_cur[i].y, 0u, 0x4140), __byte_perm(b_cur[i].y, 0u, 0x4342)};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int sh = 6 - 2 * t;
          uint32_t h[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)  // (1024 + code) - 1025 = code - 1 = weight, exact
            h[k] = hsub2(((pr[k] >> sh) & 0x00030003u) | 0x64006400u, 0x64016401u);
          *reinterpret_cast<uint4*>(Bs + swz(BN, n, 4 * t + j)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&full[st]);
    }
  } else if (lane == 0) {
    // ---------------- MMA issue (one thread) ----------------
    const uint32_t sbase = smem_addr(smem);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb & 1;
      if (!*abort_flag && !mbar_wait_bounded(&full[st], uint32_t(kb >> 1) & 1u, err)) *abort_flag = 1;
      tc_fence_after();
      const uint32_t a0 = sbase + st * kStageBytes, b0 = a0 + kAStage;
      if (!*abort_flag) {
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint32_t off_a = (ks >> 2) * (BM * 128) + (ks & 3) * 32;
          const uint32_t off_b = (ks >> 2) * (BN * 128) + (ks & 3) * 32;
          umma_f16(tmem, umma_desc_sw128(a0 + off_a), umma_desc_sw128(b0 + off_b), kIdesc, (kb | ks) != 0);
        }
      }
      umma_commit(&empty[st]);
    }
    umma_commit(accum);
  }

  // ---------------- epilogue: warps 0-3, TMEM lanes 32w..32w+31 ----------------
  if (warp < 4) {
    if (!mbar_wait_bounded(accum, 0, err)) *abort_flag = 1;
    tc_fence_after();
    const int r = warp * 32 + lane;
    const int m = m0 + r;
    const float sm = (m < M) ? s[m] : 0.f;
    const float sw = *reinterpret_cast<const float*>(packed + int64_t(N) * row_bytes);
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c), v);
      tmem_ld_wait();
      if (m < M && !*abort_flag) {
        float* yr = y + int64_t(m) * N + n0 + c;
        int32_t* ar = acc_out ? acc_out + int64_t(m) * N + n0 + c : nullptr;
        if (n0 + c + 16 <= N && (N & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            float4 o;
            o.x = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
            o.y = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 1]), sm), sw);
            o.z = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 2]), sm), sw);
            o.w = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 3]), sm), sw);
            *reinterpret_cast<float4*>(yr + j) = o;
            if (ar)
              *reinterpret_cast<int4*>(ar + j) =
                  make_int4(__float2int_rn(__uint_as_float(v[j])), __float2int_rn(__uint_as_float(v[j + 1])),
                            __float2int_rn(__uint_as_float(v[j + 2])), __float2int_rn(__uint_as_float(v[j + 3])));
          }
        } else {
          for (int j = 0; j < 16; ++j) {
            if (n0 + c + j >= N) break;
            yr[j] = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
            if (ar) ar[j] = __float2int_rn(__uint_as_float(v[j]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
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
