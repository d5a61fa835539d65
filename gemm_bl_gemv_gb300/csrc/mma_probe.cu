// Throughput probe of the warp-level int8 MMA (mma.sync m16n8k32, s8 x s8 ->
// s32).  The exact-integer products of this library run on the tcgen05 fp16
// pipe; this probe gives the rate of the legacy integer MMA path as a second
// denominator for them.  The work is register-only: four independent
// accumulator chains per warp, and each thread writes one int at the end so
// that nothing is optimised away.
#include "bl_internal.h"

namespace bl {
namespace {

constexpr int kProbeThreads = 256;

__global__ void __launch_bounds__(kProbeThreads) mma_s8_probe_kernel(int iters, int32_t* __restrict__ out) {
  const uint32_t t = threadIdx.x + 1u, b = blockIdx.x + 1u;
  const uint32_t a0 = t * 0x01010101u, a1 = a0 ^ 0x5a5a5a5au, a2 = a0 + b, a3 = ~a0;
  const uint32_t b0 = b * 0x00010203u, b1 = b0 ^ t;
  int32_t c[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) c[j][k] = 0;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int32_t s = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) s += c[j][k];
  out[int64_t(blockIdx.x) * kProbeThreads + threadIdx.x] = s;
}

}  // namespace

cudaError_t launch_mma_s8_probe(int iters, int32_t* out, int64_t out_len, int64_t* ops, cudaStream_t st) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mma_s8_probe_kernel, kProbeThreads, 0);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(int64_t(sm_count()) * std::max(per_sm, 1), out_len / kProbeThreads);
  if (grid < 1) return cudaErrorInvalidValue;
  // 2 * 16 * 8 * 32 integer operations per warp-level MMA, four per loop trip
  *ops = grid * (kProbeThreads / 32) * int64_t(iters) * 4 * (2 * 16 * 8 * 32);
  return launch(mma_s8_probe_kernel, dim3(unsigned(grid)), dim3(kProbeThreads), 0, st, false, iters, out);
}

}  // namespace bl
