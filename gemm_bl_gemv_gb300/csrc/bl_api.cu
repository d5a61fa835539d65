// C ABI of libbl: argument checks (before any launch), status codes, the
// device error word and the overlap switch.  Every product and conversion is
// done by the kernels in the other translation units.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "bl.h"
#include "bl_internal.h"

namespace bl {

// The library's device error word (BL_DEVERR_* bits).
__device__ unsigned int g_dev_error = 0;

std::atomic<unsigned long long> g_wait_limit{0};
unsigned long long wait_limit_ns() { return g_wait_limit.load(); }

namespace {
std::atomic<int> g_overlap{0};
thread_local char g_msg[512] = "";

bl_status fail(bl_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
bl_status fail(bl_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

bl_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return BL_OK;
  return fail(BL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Status of a product launcher.  The launchers return cudaErrorInvalidConfiguration
// or cudaErrorNotSupported, before any CUDA call, when a shape passed the checks
// here but no launch plan exists for it: a tile, the activation records or x do not
// fit in a CTA's shared memory, or no tensor map describes the operands.
bl_status launch_status(cudaError_t e, const char* what) {
  if (e == cudaErrorInvalidConfiguration || e == cudaErrorNotSupported)
    return fail(BL_ERR_UNSUPPORTED, "%s: no launch plan for this shape (shared memory or tensor map limits)", what);
  return cuda_status(e, what);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t S(bl_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }
}  // namespace

bool overlap_enabled() { return g_overlap.load(std::memory_order_relaxed) != 0; }

bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                       uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<Encode>(fn);
  });
  if (!encode || box_inner % 16 || box_inner == 0 || box_inner > 256 || box_outer == 0 || box_outer > 256 ||
      row_bytes % 16 || inner == 0 || outer == 0 || inner >= (uint64_t(1) << 32) || outer >= (uint64_t(1) << 32))
    return false;
  const cuuint64_t dim[2] = {inner, outer}, stride[1] = {row_bytes};
  const cuuint32_t boxd[2] = {box_inner, box_outer}, estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dim, stride, boxd, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned int* dev_error_ptr() {
  static unsigned int* cache[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) == cudaSuccess) cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

cudaError_t raise_smem_cap_impl(const void* kernel, int dev, int bytes) {
  struct Entry {
    const void* k;
    int dev, bytes;
  };
  static Entry entries[256];
  static int n = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (entries[i].k == kernel && entries[i].dev == dev && entries[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 256) entries[n++] = Entry{kernel, dev, bytes};
  return e;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

}  // namespace bl

using namespace bl;

extern "C" {

const char* bl_status_string(bl_status s) {
  switch (s) {
    case BL_OK: return "BL_OK";
    case BL_ERR_NULL: return "BL_ERR_NULL";
    case BL_ERR_SHAPE: return "BL_ERR_SHAPE";
    case BL_ERR_ALIGN: return "BL_ERR_ALIGN";
    case BL_ERR_DTYPE: return "BL_ERR_DTYPE";
    case BL_ERR_UNSUPPORTED: return "BL_ERR_UNSUPPORTED";
    case BL_ERR_CUDA: return "BL_ERR_CUDA";
  }
  return "BL_UNKNOWN_STATUS";
}

const char* bl_last_error(void) { return g_msg; }

bl_status bl_device_error(uint32_t* flags, int clear) {
  if (!flags) return fail(BL_ERR_NULL, "bl_device_error: flags is NULL");
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, bl::g_dev_error, sizeof(v));
  if (e != cudaSuccess) return cuda_status(e, "bl_device_error read");
  *flags = v;
  if (clear) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(bl::g_dev_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_status(e, "bl_device_error clear");
  }
  return BL_OK;
}

bl_status bl_set_wait_limit(uint64_t ns) {
  bl::g_wait_limit.store(ns);
  return BL_OK;
}

void bl_set_overlap(int enable) { g_overlap.store(enable ? 1 : 0); }
int bl_get_overlap(void) { return g_overlap.load(); }

bl_status bl_pack_i2s(const int8_t* w, float scale, int64_t N, int64_t K, uint8_t* out, bl_stream_t stream) {
  if (!w || !out) return fail(BL_ERR_NULL, "bl_pack_i2s: NULL pointer");
  if (N < 1 || K < 128 || K % 128) return fail(BL_ERR_SHAPE, "bl_pack_i2s: need N >= 1, K %% 128 == 0 (N=%lld K=%lld)",
                                               (long long)N, (long long)K);
  if (!aligned(out, 16)) return fail(BL_ERR_ALIGN, "bl_pack_i2s: out must be 16-byte aligned");
  return cuda_status(launch_pack_i2s(w, scale, N, K, out, S(stream)), "bl_pack_i2s");
}

bl_status bl_pack_tq2_0(const int8_t* w, const uint16_t* d_fp16, int64_t N, int64_t K, uint8_t* out,
                        bl_stream_t stream) {
  if (!w || !d_fp16 || !out) return fail(BL_ERR_NULL, "bl_pack_tq2_0: NULL pointer");
  if (N < 1 || K < 256 || K % 256)
    return fail(BL_ERR_SHAPE, "bl_pack_tq2_0: need N >= 1, K %% 256 == 0 (N=%lld K=%lld)", (long long)N, (long long)K);
  if (!aligned(out, 2) || !aligned(d_fp16, 2)) return fail(BL_ERR_ALIGN, "bl_pack_tq2_0: out and d must be 2-byte aligned");
  return cuda_status(launch_pack_tq2_0(w, d_fp16, N, K, out, S(stream)), "bl_pack_tq2_0");
}

bl_status bl_pack_w1(const int8_t* w, int64_t N, int64_t K, int32_t* out, bl_stream_t stream) {
  if (!w || !out) return fail(BL_ERR_NULL, "bl_pack_w1: NULL pointer");
  if (N < 1 || K < 32 || K % 32)
    return fail(BL_ERR_SHAPE, "bl_pack_w1: need N >= 1, K %% 32 == 0 (N=%lld K=%lld)", (long long)N, (long long)K);
  if (!aligned(out, 4)) return fail(BL_ERR_ALIGN, "bl_pack_w1: out must be 4-byte aligned");
  return cuda_status(launch_pack_w1(w, N, K, out, S(stream)), "bl_pack_w1");
}

bl_status bl_quantize_act_absmax_int8(const void* x, bl_dtype xt, int64_t M, int64_t K, int8_t* q, float* s,
                                      bl_stream_t stream) {
  if (!x || !q || !s) return fail(BL_ERR_NULL, "bl_quantize_act_absmax_int8: NULL pointer");
  if (xt != BL_F32 && xt != BL_BF16) return fail(BL_ERR_DTYPE, "bl_quantize_act_absmax_int8: bad dtype %d", int(xt));
  if (M < 1 || K < 1 || M > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_quantize_act_absmax_int8: need M >= 1, K >= 1 (M=%lld K=%lld)", (long long)M,
                (long long)K);
  if (!aligned(x, xt == BL_F32 ? 4 : 2) || !aligned(s, 4))
    return fail(BL_ERR_ALIGN, "bl_quantize_act_absmax_int8: x and s must be aligned to their element size");
  return cuda_status(launch_act_quant(x, xt, M, K, q, s, S(stream)), "bl_quantize_act_absmax_int8");
}

static bl_status check_gemv_i2s(const char* fn, const uint8_t* packed, const void* x, bl_dtype xt, const void* y,
                                bl_dtype yt, int64_t N, int64_t K) {
  if (!packed || !x || !y) return fail(BL_ERR_NULL, "%s: NULL pointer", fn);
  if ((xt != BL_F32 && xt != BL_BF16) || (yt != BL_F32 && yt != BL_BF16))
    return fail(BL_ERR_DTYPE, "%s: bad dtype (x %d, y %d)", fn, int(xt), int(yt));
  if (N < 1 || K < 128 || K % 128 || N > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "%s: need N >= 1, K %% 128 == 0 (N=%lld K=%lld)", fn, (long long)N, (long long)K);
  if (K > 32768) return fail(BL_ERR_UNSUPPORTED, "%s: K up to 32768 supported (K=%lld)", fn, (long long)K);
  if (!aligned(packed, 16)) return fail(BL_ERR_ALIGN, "%s: packed must be 16-byte aligned", fn);
  if (!aligned(x, xt == BL_F32 ? 4 : 2) || !aligned(y, yt == BL_F32 ? 4 : 2))
    return fail(BL_ERR_ALIGN, "%s: x and y must be aligned to their element size", fn);
  return BL_OK;
}

bl_status bl_gemv_i2s(const uint8_t* packed, const void* x, bl_dtype xt, void* y, bl_dtype yt, int64_t N, int64_t K,
                      bl_stream_t stream) {
  const bl_status st = check_gemv_i2s("bl_gemv_i2s", packed, x, xt, y, yt, N, K);
  if (st != BL_OK) return st;
  return launch_status(launch_gemv_i2s(packed, x, xt, y, yt, N, K, S(stream)), "bl_gemv_i2s");
}

bl_status bl_gemv_i2s_residual(const uint8_t* packed, const void* x, bl_dtype xt, const void* residual, void* y,
                               bl_dtype yt, int64_t N, int64_t K, bl_stream_t stream) {
  const bl_status st = check_gemv_i2s("bl_gemv_i2s_residual", packed, x, xt, y, yt, N, K);
  if (st != BL_OK) return st;
  if (!residual) return fail(BL_ERR_NULL, "bl_gemv_i2s_residual: residual is NULL");
  if (!aligned(residual, yt == BL_F32 ? 4 : 2))
    return fail(BL_ERR_ALIGN, "bl_gemv_i2s_residual: residual must be aligned to its element size");
  return launch_status(launch_gemv_i2s(packed, x, xt, y, yt, N, K, S(stream), residual, nullptr, 0.f),
                       "bl_gemv_i2s_residual");
}

bl_status bl_gemv_i2s_rmsnorm(const uint8_t* packed, const void* x, bl_dtype xt, const void* rms_weight, float eps,
                              const void* residual, void* y, bl_dtype yt, int64_t N, int64_t K, bl_stream_t stream) {
  const bl_status st = check_gemv_i2s("bl_gemv_i2s_rmsnorm", packed, x, xt, y, yt, N, K);
  if (st != BL_OK) return st;
  if (!rms_weight) return fail(BL_ERR_NULL, "bl_gemv_i2s_rmsnorm: rms_weight is NULL");
  if (!aligned(rms_weight, xt == BL_F32 ? 4 : 2) || (residual && !aligned(residual, yt == BL_F32 ? 4 : 2)))
    return fail(BL_ERR_ALIGN, "bl_gemv_i2s_rmsnorm: rms_weight / residual must be aligned to their element size");
  if (!(eps >= 0.f)) return fail(BL_ERR_SHAPE, "bl_gemv_i2s_rmsnorm: eps must be >= 0");
  return launch_status(launch_gemv_i2s(packed, x, xt, y, yt, N, K, S(stream), residual, rms_weight, eps),
                       "bl_gemv_i2s_rmsnorm");
}

bl_status bl_gemv_i2s_gate_up(const uint8_t* packed_gate, const uint8_t* packed_up, const void* x, bl_dtype xt,
                              void* h, bl_dtype ht, int64_t N, int64_t K, bl_stream_t stream) {
  if (!packed_gate || !packed_up || !x || !h) return fail(BL_ERR_NULL, "bl_gemv_i2s_gate_up: NULL pointer");
  if ((xt != BL_F32 && xt != BL_BF16) || (ht != BL_F32 && ht != BL_BF16))
    return fail(BL_ERR_DTYPE, "bl_gemv_i2s_gate_up: bad dtype (x %d, h %d)", int(xt), int(ht));
  if (N < 1 || K < 128 || K % 128 || N > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemv_i2s_gate_up: need N >= 1, K %% 128 == 0 (N=%lld K=%lld)", (long long)N,
                (long long)K);
  if (K > 32768) return fail(BL_ERR_UNSUPPORTED, "bl_gemv_i2s_gate_up: K up to 32768 supported (K=%lld)", (long long)K);
  if (!aligned(packed_gate, 16) || !aligned(packed_up, 16))
    return fail(BL_ERR_ALIGN, "bl_gemv_i2s_gate_up: packed tensors must be 16-byte aligned");
  if (!aligned(x, xt == BL_F32 ? 4 : 2) || !aligned(h, ht == BL_F32 ? 4 : 2))
    return fail(BL_ERR_ALIGN, "bl_gemv_i2s_gate_up: x and h must be aligned to their element size");
  return launch_status(launch_gemv_i2s_gate_up(packed_gate, packed_up, x, xt, h, ht, N, K, S(stream)),
                       "bl_gemv_i2s_gate_up");
}

bl_status bl_gemv_tq2_0(const uint8_t* packed, const void* x, bl_dtype xt, float* y, int64_t N, int64_t K,
                        bl_stream_t stream) {
  if (!packed || !x || !y) return fail(BL_ERR_NULL, "bl_gemv_tq2_0: NULL pointer");
  if (xt != BL_F32 && xt != BL_BF16) return fail(BL_ERR_DTYPE, "bl_gemv_tq2_0: bad dtype %d", int(xt));
  if (N < 1 || K < 256 || K % 256 || N > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemv_tq2_0: need N >= 1, K %% 256 == 0 (N=%lld K=%lld)", (long long)N, (long long)K);
  if (K / 256 > 1024) return fail(BL_ERR_UNSUPPORTED, "bl_gemv_tq2_0: K up to 262144 supported (K=%lld)", (long long)K);
  if (!aligned(packed, 16)) return fail(BL_ERR_ALIGN, "bl_gemv_tq2_0: packed must be 16-byte aligned");
  if (!aligned(x, xt == BL_F32 ? 4 : 2) || !aligned(y, 4))
    return fail(BL_ERR_ALIGN, "bl_gemv_tq2_0: x and y must be aligned to their element size");
  return launch_status(launch_gemv_tq2_0(packed, x, xt, y, N, K, S(stream)), "bl_gemv_tq2_0");
}

bl_status bl_gemm_w1a8(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws_fp16,
                       const uint16_t* bias_bf16, int64_t M, int64_t N, int64_t K, int group, uint16_t* y_bf16,
                       int32_t* group_dots, bl_stream_t stream) {
  if (!q || !s || !wq || !ws_fp16 || !y_bf16) return fail(BL_ERR_NULL, "bl_gemm_w1a8: NULL pointer");
  if (M < 1 || M > 0x7fffffff) return fail(BL_ERR_SHAPE, "bl_gemm_w1a8: need M >= 1 (M=%lld)", (long long)M);
  if (M > 8 && group_dots)
    return fail(BL_ERR_UNSUPPORTED, "bl_gemm_w1a8: group_dots only for M <= 8 (M=%lld)", (long long)M);
  if (M > 8 && (K % 128 || K > 132096))
    return fail(BL_ERR_UNSUPPORTED, "bl_gemm_w1a8: M > 8 needs K %% 128 == 0 and K <= 132096 (K=%lld)", (long long)K);
  if (N < 1 || K < 32 || K % 32 || group < 32 || group % 32 || K % group || N > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemm_w1a8: need N >= 1, K %% 32 == 0, group %% 32 == 0, K %% group == 0 "
                "(N=%lld K=%lld group=%d)", (long long)N, (long long)K, group);
  if (K / group > 1024) return fail(BL_ERR_UNSUPPORTED, "bl_gemm_w1a8: at most 1024 groups per row");
  if (!aligned(q, 16) || !aligned(wq, 16) || !aligned(ws_fp16, 16) || !aligned(s, 4) || !aligned(y_bf16, 2) ||
      (bias_bf16 && !aligned(bias_bf16, 2)) || (group_dots && !aligned(group_dots, 4)))
    return fail(BL_ERR_ALIGN, "bl_gemm_w1a8: q, wq, ws must be 16-byte aligned; others to their element size");
  return launch_status(launch_gemm_w1a8(q, s, wq, ws_fp16, bias_bf16, M, N, K, group, y_bf16, group_dots, S(stream)),
                       "bl_gemm_w1a8");
}

bl_status bl_gemm_w1a8_act(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws_fp16,
                           const uint16_t* bias_bf16, int64_t M, int64_t N, int64_t K, int group, uint16_t* y_bf16,
                           bl_stream_t stream) {
  if (!x || !wq || !ws_fp16 || !y_bf16) return fail(BL_ERR_NULL, "bl_gemm_w1a8_act: NULL pointer");
  if (xt != BL_F32 && xt != BL_BF16) return fail(BL_ERR_DTYPE, "bl_gemm_w1a8_act: bad dtype %d", int(xt));
  if (N < 1 || K < 32 || K % 32 || group < 32 || group % 32 || K % group || N > 0x7fffffff || M < 1)
    return fail(BL_ERR_SHAPE, "bl_gemm_w1a8_act: need M, N >= 1, K %% 32 == 0, group %% 32 == 0, K %% group == 0 "
                "(M=%lld N=%lld K=%lld group=%d)", (long long)M, (long long)N, (long long)K, group);
  if (M > 8)
    return fail(BL_ERR_UNSUPPORTED, "bl_gemm_w1a8_act: M <= 8 only; quantize larger batches with "
                "bl_quantize_act_absmax_int8 (M=%lld)", (long long)M);
  if (K / group > 1024) return fail(BL_ERR_UNSUPPORTED, "bl_gemm_w1a8_act: at most 1024 groups per row");
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(ws_fp16, 16) || !aligned(y_bf16, 2) ||
      (bias_bf16 && !aligned(bias_bf16, 2)))
    return fail(BL_ERR_ALIGN, "bl_gemm_w1a8_act: x, wq, ws must be 16-byte aligned; y, bias 2-byte aligned");
  return launch_status(launch_gemm_w1a8_act(x, xt, wq, ws_fp16, bias_bf16, M, N, K, group, y_bf16, S(stream)),
                       "bl_gemm_w1a8_act");
}

bl_status bl_gemm_tq2_0_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N,
                             int64_t K, float* y, bl_stream_t stream) {
  if (!q || !s || !packed || !y) return fail(BL_ERR_NULL, "bl_gemm_tq2_0_int8: NULL pointer");
  if (M < 1 || N < 1 || K < 256 || K % 256 || N > 0x7fffffff || M > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemm_tq2_0_int8: need M, N >= 1, K %% 256 == 0 (M=%lld N=%lld K=%lld)",
                (long long)M, (long long)N, (long long)K);
  if (K > (int64_t(1) << 24) || N * (K / 256) * 66 >= (int64_t(1) << 31))
    return fail(BL_ERR_UNSUPPORTED, "bl_gemm_tq2_0_int8: K <= 2^24 and a packed tensor under 2 GiB supported");
  if (!aligned(q, 16) || !aligned(s, 4) || !aligned(packed, 16) || !aligned(y, 16))
    return fail(BL_ERR_ALIGN, "bl_gemm_tq2_0_int8: q, packed and y must be 16-byte aligned, s 4-byte");
  return launch_status(launch_gemm_tq2_0_int8(q, s, packed, M, N, K, y, S(stream)), "bl_gemm_tq2_0_int8");
}

bl_status bl_gemm_i2s_int8(const int8_t* q, const float* s, const uint8_t* packed, int64_t M, int64_t N, int64_t K,
                           float* y, int32_t* acc, bl_stream_t stream) {
  if (!q || !s || !packed || !y) return fail(BL_ERR_NULL, "bl_gemm_i2s_int8: NULL pointer");
  if (M < 1 || N < 1 || K < 128 || K % 128 || N > 0x7fffffff || M > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemm_i2s_int8: need M, N >= 1, K %% 128 == 0 (M=%lld N=%lld K=%lld)", (long long)M,
                (long long)N, (long long)K);
  if (K > 131072) return fail(BL_ERR_UNSUPPORTED, "bl_gemm_i2s_int8: K <= 131072 supported (K=%lld)", (long long)K);
  if (!aligned(q, 16) || !aligned(s, 16) || !aligned(packed, 16) || !aligned(y, 16) || (acc && !aligned(acc, 16)))
    return fail(BL_ERR_ALIGN, "bl_gemm_i2s_int8: all pointers must be 16-byte aligned");
  return launch_status(launch_gemm_i2s_int8(q, s, packed, M, N, K, y, acc, S(stream)), "bl_gemm_i2s_int8");
}

bl_status bl_gemm_i2s_int8_act_noalloc(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N,
                                       int64_t K, float* y, int fuse, bl_stream_t stream) {
  if (!x || !packed || !y) return fail(BL_ERR_NULL, "bl_gemm_i2s_int8_act_noalloc: NULL pointer");
  if (xt != BL_F32 && xt != BL_BF16) return fail(BL_ERR_DTYPE, "bl_gemm_i2s_int8_act_noalloc: bad dtype %d", int(xt));
  if (M < 1 || N < 1 || K < 128 || K % 128 || N > 0x7fffffff || M > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemm_i2s_int8_act_noalloc: need M, N >= 1, K %% 128 == 0 (M=%lld N=%lld K=%lld)",
                (long long)M, (long long)N, (long long)K);
  if (K > 131072)
    return fail(BL_ERR_UNSUPPORTED, "bl_gemm_i2s_int8_act_noalloc: K <= 131072 supported (K=%lld)", (long long)K);
  if (M > (int64_t(1) << 40) / K || bl::gemm_i2s_int8_act_workspace(M, K) > bl::gemm_i2s_int8_act_noalloc_limit())
    return fail(BL_ERR_UNSUPPORTED,
                "bl_gemm_i2s_int8_act_noalloc: M=%lld, K=%lld needs more workspace than the static %zu bytes; "
                "use bl_gemm_i2s_int8_act with a workspace", (long long)M, (long long)K,
                bl::gemm_i2s_int8_act_noalloc_limit());
  if (!aligned(packed, 16) || !aligned(y, 16) || !aligned(x, xt == BL_F32 ? 4 : 2))
    return fail(BL_ERR_ALIGN, "bl_gemm_i2s_int8_act_noalloc: packed and y 16-byte, x element aligned");
  return launch_status(bl::launch_gemm_i2s_int8_act_noalloc(x, xt, packed, M, N, K, y, fuse, S(stream)),
                       "bl_gemm_i2s_int8_act_noalloc");
}

size_t bl_gemm_i2s_int8_act_workspace(int64_t M, int64_t K) {
  if (M < 1 || K < 1) return 0;
  return bl::gemm_i2s_int8_act_workspace(M, K);
}

bl_status bl_gemm_i2s_int8_act(const void* x, bl_dtype xt, const uint8_t* packed, int64_t M, int64_t N, int64_t K,
                               float* y, void* workspace, size_t workspace_bytes, int fuse, bl_stream_t stream) {
  if (!x || !packed || !y || !workspace) return fail(BL_ERR_NULL, "bl_gemm_i2s_int8_act: NULL pointer");
  if (xt != BL_F32 && xt != BL_BF16) return fail(BL_ERR_DTYPE, "bl_gemm_i2s_int8_act: bad dtype %d", int(xt));
  if (M < 1 || N < 1 || K < 128 || K % 128 || N > 0x7fffffff || M > 0x7fffffff)
    return fail(BL_ERR_SHAPE, "bl_gemm_i2s_int8_act: need M, N >= 1, K %% 128 == 0 (M=%lld N=%lld K=%lld)",
                (long long)M, (long long)N, (long long)K);
  if (K > 131072) return fail(BL_ERR_UNSUPPORTED, "bl_gemm_i2s_int8_act: K <= 131072 supported (K=%lld)", (long long)K);
  if (workspace_bytes < bl::gemm_i2s_int8_act_workspace(M, K))
    return fail(BL_ERR_SHAPE, "bl_gemm_i2s_int8_act: workspace of %zu bytes, need %zu", workspace_bytes,
                bl::gemm_i2s_int8_act_workspace(M, K));
  if (!aligned(workspace, 256) || !aligned(packed, 16) || !aligned(y, 16) || !aligned(x, xt == BL_F32 ? 4 : 2))
    return fail(BL_ERR_ALIGN, "bl_gemm_i2s_int8_act: workspace 256-byte, packed and y 16-byte, x element aligned");
  return launch_status(bl::launch_gemm_i2s_int8_act(x, xt, packed, M, N, K, y, static_cast<uint8_t*>(workspace),
                                                    fuse, S(stream)),
                       "bl_gemm_i2s_int8_act");
}

}  // extern "C"
