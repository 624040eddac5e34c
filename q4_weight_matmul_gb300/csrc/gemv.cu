// q4k_gemv / q4k_gemv_multi: the decode GEMV over fp32 activations and
// BLOCK144 Q4_K weights (the kernel itself is in gemv_kernel.cuh).
#include "gemv_kernel.cuh"

namespace q4k {

int gemv_max_mats() { return kMaxMats; }

bool gemv_supported(const int64_t* rows, int n_mats, int64_t cols, int batch) {
  if (batch < 1 || batch > 8 || n_mats < 1 || n_mats > kMaxMats) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return make_plan(batch, rows, n_mats, (int)(cols / kQK), device_info(dev), false, kFmtQ4K).ring != 0;
}

cudaError_t launch_gemv_block144(const uint8_t* const* w, const int64_t* rows, int n_mats, int64_t cols,
                                 const float* x, int batch, const float* const* residual,
                                 float* const* y, cudaStream_t s) {
  const ActIn act{x, nullptr, nullptr, nullptr, nullptr};
  return launch_batch<kActF32, kFmtQ4K>(w, rows, n_mats, (int)(cols / kQK), batch, act, residual, y, s);
}

}  // namespace q4k
