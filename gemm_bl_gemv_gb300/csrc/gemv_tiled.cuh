// Tiled, TMA-staged skeleton shared by the M<=8 products (i2_s GEMV, TQ2_0
// GEMV, W1A8 small-batch GEMM).
//
// Work decomposition
//   * A row of packed weights is cut into nC "chunks", the format's natural
//     unit: a 128-element i2_s group (32 B), a 256-element TQ2_0 block (66 B)
//     or a W1 scale group (group/8 B).
//   * A CTA owns a tile of TR = P*R consecutive rows.  Thread (c, g) works on
//     chunk c of rows g*R .. g*R+R-1 of the tile, so each activation word it
//     loads from shared memory is reused for R rows.
//   * Tiles are bulk-copied (cp.async.bulk, the non-tensor TMA) from global
//     memory into a ring of `stages` shared-memory buffers; one mbarrier per
//     buffer completes on the copied byte count.  Thread 0 refills a buffer
//     as soon as every thread has finished reading it.
//   * Each thread writes one fp32 partial per (output, row, chunk) to shared
//     memory; the partials of a row are summed in chunk order by one thread,
//     so results do not depend on timing (no atomics, bitwise repeatable).
//   * Activations are converted once per CTA (before the first tile) into
//     the layout the policy needs.  With programmatic dependent launch the
//     weight copies for the first tiles are issued before waiting on the
//     previous kernel; activations are read only after that wait.
//
// A Policy provides:
//   static constexpr int kOut;          outputs per row held in partials
//   struct Args;                        kernel arguments
//   static const uint8_t* weights(const Args&);
//   static const uint8_t* aux(const Args&);   (second per-row tensor, or nullptr)
//   static void prepare(const Args&, const TileGeom&, uint8_t* smem, int tid, int T);  (block-wide, ends synced)
//   static void compute(const Args&, const TileGeom&, const uint8_t* tile, const uint8_t* smem,
//                       int c, int g, int row0, int rows, float* part);
//   static void finish(const Args&, const TileGeom&, const uint8_t* smem, const float* part,
//                      int row0, int rows, int tid, int T);
#pragma once
#include "bl_device.cuh"

namespace bl {

struct TileGeom {
  int N;                 // rows of the weight matrix
  int nC;                // chunks per row
  int P;                 // row groups per tile
  int R;                 // rows per thread
  int TR;                // rows per tile (P*R)
  int stages;            // shared-memory ring depth
  int ntiles;            // ceil(N / TR)
  int kout;              // outputs per row (tokens)
  int64_t row_bytes;     // packed bytes per row
  int64_t aux_row_bytes; // bytes per row of an optional second tensor copied with the tile (0: none)
  uint32_t aux_off;      // offset of that second segment inside a ring buffer
  uint32_t stage_bytes;  // bytes of one ring buffer (multiple of 128)
  uint32_t off_bar;      // offsets into dynamic shared memory
  uint32_t off_stage;
  uint32_t off_part;
  uint32_t off_pol;      // policy area (activations, sums, constants)
  uint32_t smem_bytes;
  unsigned int* err;     // the library's device error word
};

template <class Pol>
__global__ void __launch_bounds__(Pol::kMaxThreads) tiled_kernel(typename Pol::Args a, TileGeom g, int early_weights) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  uint8_t* ring = smem + g.off_stage;
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const uint8_t* wsrc = Pol::weights(a);
  const uint8_t* asrc = Pol::aux(a);
  const int my_tiles = (int(blockIdx.x) < g.ntiles) ? (g.ntiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;

  // Issue the bulk copy of local tile i into ring buffer i % stages (thread 0).
  auto issue = [&](int i) {
    const int t = int(blockIdx.x) + i * int(gridDim.x);
    const int s = i % g.stages;
    const int64_t r0 = int64_t(t) * g.TR;
    const int64_t nr = (g.N - r0 < g.TR) ? (g.N - r0) : g.TR;
    uint8_t* dst = ring + size_t(s) * g.stage_bytes;
    const uint8_t* src = wsrc + uint64_t(r0) * uint64_t(g.row_bytes);
    const uint64_t bytes = uint64_t(nr) * uint64_t(g.row_bytes);
    const uint32_t b16 = uint32_t(bytes & ~uint64_t(15));
    // bytes past the last multiple of 16 (only possible on the last tile of
    // a matrix whose rows are not 16-byte multiples) go by plain loads
    for (uint32_t k = b16; k < uint32_t(bytes); ++k) dst[k] = src[k];
    uint32_t a16 = 0;
    const uint8_t* asrc_t = nullptr;
    uint8_t* adst = dst + g.aux_off;
    if (g.aux_row_bytes) {
      asrc_t = asrc + uint64_t(r0) * uint64_t(g.aux_row_bytes);
      const uint64_t abytes = uint64_t(nr) * uint64_t(g.aux_row_bytes);
      a16 = uint32_t(abytes & ~uint64_t(15));
      for (uint32_t k = a16; k < uint32_t(abytes); ++k) adst[k] = asrc_t[k];
    }
    mbar_arrive_expect_tx(&full[s], b16 + a16);
    const uint64_t pol = policy_evict_first();
    if (b16) bulk_g2s(dst, src, b16, &full[s], pol);
    if (a16) bulk_g2s(adst, asrc_t, a16, &full[s], pol);
  };

  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int npre = my_tiles < g.stages ? my_tiles : g.stages;
  if (early_weights && tid == 0)
    for (int i = 0; i < npre; ++i) issue(i);
  pdl_wait();
  if (!early_weights && tid == 0)
    for (int i = 0; i < npre; ++i) issue(i);

  Pol::prepare(a, g, smem, tid, T);
  pdl_launch_dependents();

  const int c = tid % g.nC;
  const int grp = tid / g.nC;
  const int part_stride = g.kout * g.TR * g.nC;
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % g.stages;
    const uint32_t parity = uint32_t(i / g.stages) & 1u;
    bool ok = mbar_wait_bounded(&full[s], parity, g.err);
    const int t = int(blockIdx.x) + i * int(gridDim.x);
    const int row0 = t * g.TR;
    const int rows = (g.N - row0 < g.TR) ? (g.N - row0) : g.TR;
    float* pb = part + (i & 1) * part_stride;
    if (ok && grp < g.P) Pol::compute(a, g, ring + size_t(s) * g.stage_bytes, smem, c, grp, row0, rows, pb);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      // A copy did not land in time: let copies still in flight finish
      // (bounded), then leave.  The error flag is already set.
      if (tid == 0)
        for (int j = i; j < my_tiles && j < i + g.stages; ++j)
          mbar_wait_bounded(&full[j % g.stages], uint32_t(j / g.stages) & 1u, nullptr);
      return;
    }
    if (tid == 0 && i + g.stages < my_tiles) issue(i + g.stages);
    Pol::finish(a, g, smem, pb, row0, rows, tid, T);
  }
}

// Shared-memory layout and launch geometry for a policy.  pol_bytes: bytes of
// the policy area.  Returns false if it does not fit.
inline bool plan_tiles(TileGeom& g, int64_t N, int nC, int P, int R, int kout, int64_t row_bytes, int stages,
                       uint32_t pol_bytes, uint32_t max_smem, int64_t aux_row_bytes = 0) {
  auto up = [](uint64_t v, uint64_t a) { return (v + a - 1) / a * a; };
  g.aux_row_bytes = aux_row_bytes;
  g.err = nullptr;
  g.N = int(N);
  g.nC = nC;
  g.P = P;
  g.R = R;
  g.TR = P * R;
  g.kout = kout;
  g.row_bytes = row_bytes;
  g.ntiles = int((N + g.TR - 1) / g.TR);
  g.aux_off = uint32_t(up(uint64_t(P * R) * uint64_t(row_bytes), 128));
  g.stage_bytes = uint32_t(up(g.aux_off + uint64_t(P * R) * uint64_t(aux_row_bytes), 128));
  for (int st = stages; st >= 2; --st) {
    uint64_t off = 0;
    g.off_bar = uint32_t(off);
    off = up(off + 8 * uint64_t(st), 128);
    g.off_stage = uint32_t(off);
    off = up(off + uint64_t(st) * g.stage_bytes, 128);
    g.off_part = uint32_t(off);
    off = up(off + 2ull * kout * g.TR * nC * 4, 128);
    g.off_pol = uint32_t(off);
    off = up(off + pol_bytes, 128);
    if (off <= max_smem) {
      g.stages = st;
      g.smem_bytes = uint32_t(off);
      return true;
    }
  }
  return false;
}

}  // namespace bl
