// W1A8 product for 1 <= M <= 8 tokens with the per-token absmax int8
// quantization fused into the prologue: the lane-per-row kernel of
// gemm_w1a8_rows.cuh, instantiated for fp32 and bf16 activations.
#include "gemm_w1a8_rows.cuh"

namespace bl {

cudaError_t launch_gemm_w1a8_act(const void* x, bl_dtype xt, const int32_t* wq, const uint16_t* ws,
                                 const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                 cudaStream_t st) {
  if (w1a8_m1_applicable(M, N, K, group)) {
    const cudaError_t e = launch_gemm_w1a8_m1(nullptr, nullptr, x, xt, wq, ws, bias, N, K, y, nullptr, st);
    if (e != cudaErrorNotSupported) return e;
  }
  if (w1a8_rows_applicable(M, K, group)) {
    const cudaError_t e =
        xt == BL_BF16 ? dispatch<false, 2>(int(M), nullptr, nullptr, x, wq, ws, bias, N, K, group, y, nullptr, st)
                      : dispatch<false, 1>(int(M), nullptr, nullptr, x, wq, ws, bias, N, K, group, y, nullptr, st);
    if (e != cudaErrorNotSupported) return e;
  }
  return launch_gemm_w1a8_act_tiled(x, xt, wq, ws, bias, M, N, K, group, y, st);
}

}  // namespace bl
