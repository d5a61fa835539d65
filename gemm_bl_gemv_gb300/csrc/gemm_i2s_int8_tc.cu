// i2_s x int8 product on the 5th-generation tensor cores (tcgen05):
//   acc[m,n] = sum_k q[m,k] w[n,k]   (exact)
//   y[m,n]   = f32(acc[m,n]) * s[m] * scale
// ("Hesper/Layers/BitLinear", "BitLinear Mathematics", with int8 activations
// from the per-token absmax quantizer).
//
// Exactness.  The MMA runs kind::f16 (fp16 operands, fp32 accumulation).
// Activations and weights enter as power-of-two multiples of q and w whose
// products are exactly q*w (see "Scaled operands" below); every partial sum
// is an integer of magnitude <= K * 128 <= 2^24 (K <= 131072), so the fp32
// accumulator holds the exact integer sum.  (This toolchain does not accept
// tcgen05 .kind::i8 for sm_103a.)
//
// Structure, one CTA per 128 x 192 output tile, K in blocks of 128 (one i2_s
// group), a 3-stage pipeline:
//   * one lane of warp 17 brings each K block's raw operands into shared
//     memory with two TMA loads: the 128 x 128 int8 activation tile
//     (128-byte swizzle) and the 192 x 32 bytes of packed weight codes;
//   * warps 0-3 take the activations to tensor memory: the thread of TMEM
//     lane r converts the 128 int8 of row r to scaled fp16 and writes 64
//     columns with tcgen05.st;
//   * warps 4-15 expand the packed weights to fp16 in shared memory, in the
//     K-major 128-byte-swizzled layout the tensor core reads.  The eight
//     lanes of a store phase hold eight rows, whose swizzle puts the same
//     chunk on eight distinct bank groups;
//   * one lane of warp 16 allocates the 512 TMEM columns (accumulator
//     0..191, activation stages from 256) and issues eight 128x192x16 MMAs
//     per K block, A from TMEM, B from shared memory; tcgen05.commit frees
//     the stage and finally signals the epilogue;
//   * warps 0-15 read the accumulator (warp w: lanes 32(w%4).., 48 columns),
//     stage y in shared memory and write each row segment with one bulk
//     copy (acc likewise when asked).
// Every wait is bounded; on a timeout the CTA records the error flag,
// finishes its loops without waiting, and still frees its TMEM.
#include "act_quant.cuh"
#include "bl_device.cuh"
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int BM = 128, BN = 192, BK = 128;
constexpr int kAWarps = 4;                    // activation warps: TMEM lane quarter w % 4, classes of w / 4
static_assert(kAWarps == 4 || kAWarps == 8, "one or two activation warps per TMEM lane quarter");
constexpr int kBWarps = 12;                   // weight decoding warps
constexpr int kProducers = 32 * (kAWarps + kBWarps);
constexpr int kBThreads = 32 * kBWarps;
constexpr int kRuns = BN * 4 / kBThreads;     // 8-byte code runs (32 elements) per decoding thread and block
static_assert(kRuns * kBThreads == BN * 4 && (kBWarps * kRuns) % 24 == 0, "runs must divide evenly");
constexpr int kMmaWarp = kAWarps + kBWarps;   // TMEM allocation, MMA issue
constexpr int kThreads = 32 * (kMmaWarp + 2);  // + one warp of TMA loads
constexpr int kEpilogue = 512;                // warps 0..15 run the epilogue
constexpr int kStages = 3;
constexpr uint32_t kBStage = BN * BK * 2;  // 48 KB: two 64-column sub-tiles of 24 KB
constexpr uint32_t kAStage = BM * BK;      // 16 KB of int8 activations, 128-byte swizzled
constexpr uint32_t kWStage = BN * BK / 4;  // 6 KB of packed codes, 32 bytes per row
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 256;                // activation stage st at columns 256 + 64 st
constexpr uint32_t kOutStride = BN * 4 + 16;   // staged output row, padded against bank conflicts
constexpr uint32_t kOutBytes = BM * kOutStride;
constexpr uint32_t kPipeBytes = kStages * kBStage;
constexpr uint32_t kDataBytes = kPipeBytes > kOutBytes ? kPipeBytes : kOutBytes;
constexpr uint32_t kAOff = kDataBytes;  // 1024-aligned (the swizzle repeats every 1024 bytes)
constexpr uint32_t kWOff = kAOff + kStages * kAStage;
constexpr uint32_t kBarOff = kWOff + kStages * kWStage;
constexpr size_t kSmem = size_t(kBarOff) + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kAcol + 64 * kStages <= kTmemCols && BN <= kAcol, "TMEM layout");
static_assert(kAOff % 1024 == 0 && kWOff % 128 == 0 && kWStage % 128 == 0, "TMA destinations");

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both
// K-major, N = 192, M = 128.  The B stage is [192 rows][128 K] fp16 as two
// 64-column sub-tiles, 128-byte swizzled: 16-byte chunk c of row n sits at
//   (c / 8) * 192 * 128 + (n / 8) * 1024 + (n % 8) * 128 + ((c % 8) ^ (n % 8)) * 16.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

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

// Workspace of the fused form: two barrier words at its start (count,
// generation), then q [M][K] at byte 256, then s [M] at the next 256 bytes.
constexpr size_t kWsQ = 256;
__host__ __device__ constexpr size_t ws_s_offset(size_t M, size_t K) { return kWsQ + (M * K + 255) / 256 * 256; }

// Fused quantization, before the product (cooperative launch: every CTA is
// resident).  The CTAs split the tokens; the warps 0-15 of a CTA take its
// tokens 16 / wpt at a time (wpt warps per token, a power of two), each
// thread taking 8-element chunks: a first sweep finds the token's absmax, a
// second (the same chunks, from L1) writes the codes.  Then a grid barrier: the last CTA to arrive resets the count and
// advances the generation the others wait on (bounded), so the workspace's
// barrier words are back in their initial state after every call.
template <bool XB>
__device__ __forceinline__ bool quantize_and_sync(const void* x, int M, int K, int8_t* q, float* sc,
                                                  unsigned int* bar, unsigned int* err) {
  __shared__ float red[16];
  const int G = int(gridDim.x * gridDim.y), cta = int(blockIdx.y * gridDim.x + blockIdx.x);
  const int t0 = int(int64_t(cta) * M / G), t1 = int(int64_t(cta + 1) * M / G);
  const int nt = t1 - t0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int wpt = 16;
  while (wpt > 1 && wpt * nt > 16) wpt >>= 1;
  const int tp = 16 / wpt;  // tokens per pass
  const int tok = warp / wpt, wi = warp % wpt;
  const int n8 = K / 8, tt = 32 * wpt, i0 = 32 * wi + lane;
  const size_t row_bytes = size_t(K) * (XB ? 2 : 4);
  for (int base = 0; base < nt; base += tp) {
    const int m = t0 + base + tok;
    const bool active = warp < 16 && base + tok < nt;
    const void* xr = reinterpret_cast<const uint8_t*>(x) + size_t(active ? m : 0) * row_bytes;
    float a = 0.f;
    if (active)
      for (int k8 = i0; k8 < n8; k8 += tt) {
        float v[8];
        load8<XB>(xr, k8, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[j]));
      }
    a = warp_max(a);
    if (warp < 16 && lane == 0) red[warp] = a;
    __syncthreads();
    if (active) {
      float amax = 0.f;
      for (int w = tok * wpt; w < (tok + 1) * wpt; ++w) amax = fmaxf(amax, red[w]);
      float s_m, inv;
      absmax_scales(amax, s_m, inv);
      if (i0 == 0) sc[m] = s_m;
      uint2* qr = reinterpret_cast<uint2*>(q + size_t(m) * K);
      for (int k8 = i0; k8 < n8; k8 += tt) {
        float v[8];
        load8<XB>(xr, k8, v);
        qr[k8] = quant8(v, inv);
      }
    }
    __syncthreads();  // red is reused by the next pass
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // the product reads q through TMA
  __syncthreads();
  __shared__ int ok;
  if (threadIdx.x == 0) {
    ok = 1;
    volatile unsigned int* vgen = bar + 1;
    const unsigned int gen = *vgen;
    __threadfence();
    if (atomicAdd(bar, 1u) == unsigned(G - 1)) {
      bar[0] = 0u;
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const unsigned long long start = globaltimer_ns();
      while (true) {
        unsigned int g;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(bar + 1) : "memory");
        if (g != gen) break;
        if (globaltimer_ns() - start > kWaitLimitNs) {
          atomicOr(err, BL_DEVERR_WAIT_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return ok != 0;
}

// XQ = 0: q and s given.  XQ = 1 (fp32 x) / 2 (bf16 x): x given; the codes
// and scales go to the workspace (ws) first, and qmap describes its q.
template <int XQ>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_i2s_int8_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                            const float* __restrict__ s, const uint8_t* __restrict__ packed, int M, int N, int K,
                            float* __restrict__ y, int32_t* __restrict__ acc_out, unsigned int* err,
                            const void* __restrict__ x, uint8_t* __restrict__ ws) {
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
  const int64_t row_bytes = K / 4;

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
  pdl_wait();
  if (XQ) {
    int8_t* wq = reinterpret_cast<int8_t*>(ws + kWsQ);
    float* ws_s = reinterpret_cast<float*>(ws + ws_s_offset(size_t(M), size_t(K)));
    if (!quantize_and_sync<XQ == 2>(x, M, K, wq, ws_s, reinterpret_cast<unsigned int*>(ws), err) &&
        threadIdx.x == 0)
      *abort_flag = 1;
    s = ws_s;
    __syncthreads();
  }

  if (warp < kAWarps) {
    // ------- activation converters: TMEM lane / tile row ra = 32 (w % 4) +
    //         lane, classes t of a block with t % (kAWarps / 4) = w / 4
    //         (TMEM columns 16t..16t+15 hold class t) -------
    constexpr int kTStep = kAWarps / 4;
    const int quarter = warp & 3, t0 = warp >> 2;
    const int ra = quarter * 32 + lane;
    const uint32_t a_taddr = tmem + (uint32_t(quarter * 32) << 16) + kAcol;
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
      for (int tt = 0; tt < 4; tt += kTStep) {  // chunks 2t, 2t+1 = class t
        const int t = tt + t0;
        const uint32_t sc = f16x2_pow2(2 * t - 6);
        const uint32_t bias = hfma2(0x64806480u, sc, 0x80008000u) ^ 0x80008000u;  // -(1152 * scale)
        uint4 v[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) v[i] = *reinterpret_cast<const uint4*>(arow + (((2 * t + i) ^ (ra & 7)) << 4));
        if (tt + kTStep == 4) mbar_arrive(&raw_empty[st]);
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 c = v[i];
          i8x4_to_f16_scaled(c.x, sc, bias, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_f16_scaled(c.y, sc, bias, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_f16_scaled(c.z, sc, bias, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_f16_scaled(c.w, sc, bias, o[8 * i + 6], o[8 * i + 7]);
        }
        tmem_st16(a_taddr + 64 * st + 16 * t, o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[st]);
    }
  } else if (warp < kMmaWarp) {
    // ------- weight decoders: run i of a thread is row n = 8 R + lane % 8
    //         (R = decoder warp + kBWarps i), code bytes 8j..8j+7 (j = lane / 8),
    //         i.e. elements 32t + 8j .. 32t + 8j + 7 of every class t -------
    const int wb = (threadIdx.x >> 5) - kAWarps;
    const int r = lane & 7, j = lane >> 3;
    const uint32_t u = uint32_t(j ^ r);  // chunk 4t + j lands in 16-byte unit u ^ 4(t % 2)
    uint32_t rofs[kRuns], sto[kRuns];
#pragma unroll
    for (int i = 0; i < kRuns; ++i) {
      const int R = wb + kBWarps * i, n = 8 * R + r;
      rofs[i] = uint32_t(n * 32 + 8 * j);
      sto[i] = uint32_t(R * 1024 + r * 128);
    }
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % kStages;
      if (kb >= kStages && !*abort_flag &&
          !mbar_wait_bounded(&empty[st], uint32_t(kb / kStages - 1) & 1u, err))
        *abort_flag = 1;
      if (!*abort_flag && !mbar_wait_bounded(&raw_full[st], uint32_t(kb / kStages) & 1u, err)) *abort_flag = 1;
      uint2 cw[kRuns];
#pragma unroll
      for (int i = 0; i < kRuns; ++i) cw[i] = *reinterpret_cast<const uint2*>(wraw + st * kWStage + rofs[i]);
      mbar_arrive(&raw_empty[st]);
      uint8_t* Bs = smem + st * kBStage;
#pragma unroll
      for (int i = 0; i < kRuns; ++i) {
        // code byte p of the run spread so that it lands in an fp16 half
        const uint32_t pr[4] = {__byte_perm(cw[i].x, 0u, 0x4140), __byte_perm(cw[i].x, 0u, 0x4342),
                                __byte_perm(cw[i].y, 0u, 0x4140), __byte_perm(cw[i].y, 0u, 0x4342)};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t mask = 0x00030003u << (6 - 2 * t);
          const uint32_t off = 0x64006400u | (0x00010001u << (6 - 2 * t));  // 1024 + 2^(6-2t)
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = hsub2((pr[k] & mask) | 0x64006400u, off);
          const uint32_t unit = u ^ uint32_t(4 * (t & 1));
          *reinterpret_cast<uint4*>(Bs + (t >> 1) * (BN * 128) + sto[i] + (unit << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&full[st]);
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
      tma_load_2d(wraw + st * kWStage, &wmap, kb * (BK / 4), n0, &raw_full[st]);
      issued = kb + 1;
    }
    // the CTA must not finish while a load still writes its shared memory
    for (int kb = issued - kStages < 0 ? 0 : issued - kStages; kb < issued; ++kb)
      mbar_wait_bounded(&raw_full[kb % kStages], uint32_t(kb / kStages) & 1u, nullptr);
  }

  // ------- epilogue: warps 0-15; warp w reads TMEM lanes 32(w%4).. (its rows)
  //         and columns 48(w/4) .. 48(w/4)+47, 16 at a time -------
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
    const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(c0);
    if ((N & 3) == 0) {
      // stage the tile in shared memory (the operand stages are free now) and
      // write each row segment with one bulk copy
      const int ncols = min(BN, N - n0);
      float* stage_row = reinterpret_cast<float*>(smem + r * kOutStride) + c0;
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        uint32_t v[16];
        tmem_ld16(trow + 16 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 o;
          o.x = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
          o.y = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 1]), sm), sw);
          o.z = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 2]), sm), sw);
          o.w = __fmul_rn(__fmul_rn(__uint_as_float(v[j + 3]), sm), sw);
          *reinterpret_cast<float4*>(stage_row + 16 * g + j) = o;
        }
      }
      fence_async_smem();
      named_barrier_sync(1, kEpilogue);
      const bool issuer = threadIdx.x < BM && m0 + int(threadIdx.x) < M && ok;
      if (issuer) {
        bulk_s2g(y + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride, uint32_t(ncols) * 4);
        bulk_commit();
      }
      if (acc_out) {
        if (issuer) bulk_wait_read();
        named_barrier_sync(1, kEpilogue);
        int* stage_acc = reinterpret_cast<int*>(smem + r * kOutStride) + c0;
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          uint32_t v[16];
          tmem_ld16(trow + 16 * g, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<int4*>(stage_acc + 16 * g + j) =
                make_int4(__float2int_rn(__uint_as_float(v[j])), __float2int_rn(__uint_as_float(v[j + 1])),
                          __float2int_rn(__uint_as_float(v[j + 2])), __float2int_rn(__uint_as_float(v[j + 3])));
        }
        fence_async_smem();
        named_barrier_sync(1, kEpilogue);
        if (issuer) {
          bulk_s2g(acc_out + int64_t(m0 + threadIdx.x) * N + n0, smem + threadIdx.x * kOutStride,
                   uint32_t(ncols) * 4);
          bulk_commit();
        }
      }
      if (issuer) bulk_wait_read();  // the global writes complete with the grid
    } else {
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        uint32_t v[16];
        tmem_ld16(trow + 16 * g, v);  // warp-collective: every lane loads, only rows below M store
        tmem_ld_wait();
        if (m < M && ok)
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + c0 + 16 * g + j;
            if (n < N) {
              y[int64_t(m) * N + n] = __fmul_rn(__fmul_rn(__uint_as_float(v[j]), sm), sw);
              if (acc_out) acc_out[int64_t(m) * N + n] = __float2int_rn(__uint_as_float(v[j]));
            }
          }
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
  pdl_launch_dependents();
}

}  // namespace

// Tensor-core path: M >= 64 (smaller batches use the CUDA-core kernel).
cudaError_t launch_gemm_i2s_int8(const int8_t* q, const float* sc, const uint8_t* packed, int64_t M, int64_t N,
                                 int64_t K, float* y, int32_t* acc, cudaStream_t s) {
  if (M < 64) return launch_gemm_i2s_int8_simt(q, sc, packed, M, N, K, y, acc, s);
  int dev = 0;
  cudaGetDevice(&dev);
  CUtensorMap qmap, wmap;  // q as [M][K] bytes (128 x 128 boxes, swizzled); codes as [N][K/4] bytes (192 x 32)
  if (!encode_tmap_2d_u8(&qmap, q, uint64_t(K), uint64_t(M), uint64_t(K), BK, BM, true) ||
      !encode_tmap_2d_u8(&wmap, packed, uint64_t(K / 4), uint64_t(N), uint64_t(K / 4), BK / 4, BN, false))
    return cudaErrorNotSupported;
  cudaError_t e = raise_smem_cap(gemm_i2s_int8_tc_kernel<0>, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  return launch(gemm_i2s_int8_tc_kernel<0>, grid, dim3(kThreads), kSmem, s, overlap_enabled(), qmap, wmap, sc, packed,
                int(M), int(N), int(K), y, acc, dev_error_ptr(), static_cast<const void*>(nullptr),
                static_cast<uint8_t*>(nullptr));
}

size_t gemm_i2s_int8_act_workspace(int64_t M, int64_t K) {
  return ws_s_offset(size_t(M), size_t(K)) + (size_t(M) * 4 + 255) / 256 * 256;
}

// The product from unquantized x: act-quant into the workspace, then the
// product (two launches); with `fuse`, one cooperative launch (quantization,
// grid barrier, product) when every CTA fits on the GPU at once and x's rows
// are 16-byte aligned with K % 8 == 0.
cudaError_t launch_gemm_i2s_int8_act(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                     int64_t K, float* y, uint8_t* ws, int fuse, cudaStream_t s) {
  int8_t* q = reinterpret_cast<int8_t*>(ws + kWsQ);
  float* sc = reinterpret_cast<float*>(ws + ws_s_offset(size_t(M), size_t(K)));
  const bool xb = xt == BL_BF16;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  const bool one = fuse && M >= 64 && K % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (K * (xb ? 2 : 4)) % 16 == 0 && tiles <= sm_count();
  if (!one) {
    cudaError_t e = launch_act_quant(x, xt, M, K, q, sc, s);
    if (e != cudaSuccess) return e;
    return launch_gemm_i2s_int8(q, sc, packed, M, N, K, y, nullptr, s);
  }
  int dev = 0;
  cudaGetDevice(&dev);
  CUtensorMap qmap, wmap;
  if (!encode_tmap_2d_u8(&qmap, q, uint64_t(K), uint64_t(M), uint64_t(K), BK, BM, true) ||
      !encode_tmap_2d_u8(&wmap, packed, uint64_t(K / 4), uint64_t(N), uint64_t(K / 4), BK / 4, BN, false))
    return cudaErrorNotSupported;
  auto kern = xb ? gemm_i2s_int8_tc_kernel<2> : gemm_i2s_int8_tc_kernel<1>;
  cudaError_t e = raise_smem_cap(kern, dev, int(kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, qmap, wmap, static_cast<const float*>(nullptr), packed, int(M), int(N),
                            int(K), y, static_cast<int32_t*>(nullptr), dev_error_ptr(), x, ws);
}

}  // namespace bl
