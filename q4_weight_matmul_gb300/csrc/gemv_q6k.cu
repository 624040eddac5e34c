// q6k_gemv: the decode GEMV kernel over fp32 activations and GPU-layout
// Q6_K weights (genie-ai-runtime §6, Path G: the Q6_K layout redesigned for
// vectorised loads; layout in q6k_pack.cu, superblock dot in gemv_common.cuh).
#include "gemv_kernel.cuh"

namespace q4k {

bool gemv_q6k_supported(int64_t rows, int64_t cols, int batch) {
  if (batch < 1 || batch > 8) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return make_plan(batch, &rows, 1, (int)(cols / kQK), device_info(dev), false, kFmtQ6K).ring != 0;
}

cudaError_t launch_gemv_q6k(const uint8_t* w, int64_t rows, int64_t cols, const float* x, int batch,
                            const float* residual, float* y, cudaStream_t s) {
  const ActIn act{x, nullptr, nullptr, nullptr, nullptr};
  const uint8_t* const ws[1] = {w};
  const float* const res[1] = {residual};
  float* const ys[1] = {y};
  return launch_batch<kActF32, kFmtQ6K>(ws, &rows, 1, (int)(cols / kQK), batch, act, res, ys, s);
}

}  // namespace q4k
