// W1A8 product for 1 <= M <= 8 tokens with int8 activations given: the
// lane-per-row kernel of gemm_w1a8_rows.cuh, instantiated for q and s.
#include "gemm_w1a8_rows.cuh"

namespace bl {

// The lane-per-row kernel applies when every row slice is 16-byte aligned.
bool w1a8_rows_applicable(int64_t M, int64_t K, int G) {
  return M >= 1 && M <= 8 && K % 128 == 0 && (K / G) % 8 == 0 && G <= 256;
}

cudaError_t launch_gemm_w1a8_rows(const int8_t* q, const float* s, const int32_t* wq, const uint16_t* ws,
                                  const uint16_t* bias, int64_t M, int64_t N, int64_t K, int group, uint16_t* y,
                                  int32_t* dots, cudaStream_t st) {
  if (dots) return dispatch<true, 0>(int(M), q, s, nullptr, wq, ws, bias, N, K, group, y, dots, st);
  return dispatch<false, 0>(int(M), q, s, nullptr, wq, ws, bias, N, K, group, y, dots, st);
}

}  // namespace bl
