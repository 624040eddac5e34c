// q6k_gemv_q8 (and q6k_gemm): the decode GEMV kernel over GPU-layout Q6_K
// weights and q8_1 activations, int8 or binary16 quants (the MMQ form:
// exact per-16-weight group dots, superblock_dot_q6_q8 in gemv_common.cuh).
#include "gemv_kernel.cuh"

namespace q4k {

bool gemv_q6k_q8_supported(int64_t rows, int64_t cols, int batch) {
  if (batch < 1 || batch > 8) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return make_plan(batch, &rows, 1, (int)(cols / kQK), device_info(dev), true, kFmtQ6K).ring != 0;
}

cudaError_t launch_gemv_q6k_q8(const uint8_t* w, int64_t rows, int64_t cols, const void* q8, bool h16,
                               const float* d8, const int32_t* sum, int batch, const float* residual, float* y,
                               int32_t* p_out, cudaStream_t s) {
  const ActIn act{nullptr, q8, d8, sum, p_out};
  const uint8_t* const ws[1] = {w};
  const float* const res[1] = {residual};
  float* const ys[1] = {y};
  const int nb = (int)(cols / kQK);
  return h16 ? launch_batch<kActQ8H, kFmtQ6K>(ws, &rows, 1, nb, batch, act, res, ys, s)
             : launch_batch<kActQ8, kFmtQ6K>(ws, &rows, 1, nb, batch, act, res, ys, s);
}

}  // namespace q4k
