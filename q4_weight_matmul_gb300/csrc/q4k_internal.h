// Internal declarations shared by the library's translation units.
// Launchers validate nothing: the C-ABI layer (abi.cu) checks every argument
// before it calls one.  Each returns the cudaError_t of its launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

struct q4k_gemv_job;

namespace q4k {

constexpr int kQK = 256;         // weights per superblock
constexpr int kSub = 32;         // weights per sub-block
constexpr int kBlockBytes = 144; // bytes of one BLOCK144 superblock
constexpr int kQ6GgufBytes = 210;  // bytes of one GGUF Q6_K superblock
constexpr int kQ6GpuBytes = 208;   // bytes of one GPU-layout Q6_K superblock (d kept apart)

// Device properties the launchers size their grids by (cached per device).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;   // bytes of dynamic shared memory a CTA may opt into
  int l2_bytes;
};
const DeviceInfo& device_info(int device);

// Library-owned device error word of the current device (see abi.cu).
int* device_error_word();

cudaError_t launch_pack_block144(const uint16_t* d, const uint16_t* dmin,
                                 const uint8_t* sc, const uint8_t* m,
                                 const uint8_t* q, int64_t rows, int64_t cols,
                                 uint8_t* w, cudaStream_t s);

cudaError_t launch_unpack_block144(const uint8_t* w, int64_t rows, int64_t cols, uint16_t* d, uint16_t* dmin,
                                   uint8_t* sc, uint8_t* m, uint8_t* q, cudaStream_t s);

cudaError_t launch_q8_quantize(const float* x, int64_t tokens, int64_t cols,
                               int8_t* q, float* d8, int32_t* sum,
                               cudaStream_t s);
// The same quantisation with the quants stored as exact binary16 integers.
cudaError_t launch_q8_quantize_h16(const float* x, int64_t tokens, int64_t cols, uint16_t* q, float* d8,
                                   int32_t* sum, cudaStream_t s);

// Decode GEMV over n_mats (1..gemv_max_mats()) matrices that share one input
// x; matrix m has rows[m] rows, output y[m] and optional residual[m].
// Returns cudaErrorNotSupported when the shape does not fit the kernel's
// shared-memory staging of the activations.
int gemv_max_mats();
cudaError_t launch_gemv_block144(const uint8_t* const* w, const int64_t* rows, int n_mats, int64_t cols,
                                 const float* x, int batch, const float* const* residual,
                                 float* const* y, cudaStream_t s);
bool gemv_supported(const int64_t* rows, int n_mats, int64_t cols, int batch);
// The same kernel over q8_1 activations (batch 1..8 tokens), int8 quants or
// (h16) binary16 integers; p_out (nullable) receives the exact block dots
// [batch][rows][cols/32].
bool gemv_q8_supported(int64_t rows, int64_t cols, int batch);
cudaError_t launch_gemv_q8_block144(const uint8_t* w, int64_t rows, int64_t cols, const void* q8, bool h16,
                                    const float* d8, const int32_t* sum, int batch, const float* residual,
                                    float* y, int32_t* p_out, cudaStream_t s);

// Q6_K: bytes of one row in the GPU layout (nb superblocks), conversions
// between fields (in_layout / out_layout -1), GGUF (0) and GPU (1) bytes,
// and the decode GEMV over the GPU layout.
int64_t q6k_gpu_row_bytes(int64_t nb);
cudaError_t launch_q6k_convert(const uint16_t* d_in, const int8_t* sc_in, const uint8_t* q_in, const uint8_t* w_in,
                               int in_layout, int64_t rows, int64_t cols, uint16_t* d_out, int8_t* sc_out,
                               uint8_t* q_out, uint8_t* w_out, int out_layout, cudaStream_t s);
bool gemv_q6k_supported(int64_t rows, int64_t cols, int batch);
cudaError_t launch_gemv_q6k(const uint8_t* w, int64_t rows, int64_t cols, const float* x, int batch,
                            const float* residual, float* y, cudaStream_t s);
// The same over q8_1 activations (MMQ form, 1..8 tokens); p_out (nullable)
// receives the exact 16-weight group dots [batch][rows][cols/16].
bool gemv_q6k_q8_supported(int64_t rows, int64_t cols, int batch);
cudaError_t launch_gemv_q6k_q8(const uint8_t* w, int64_t rows, int64_t cols, const void* q8, bool h16,
                               const float* d8, const int32_t* sum, int batch, const float* residual, float* y,
                               int32_t* p_out, cudaStream_t s);

// Persistent GEMV over an ordered job list (q4k_gemv_seq).  Both return a
// q4k_status; launch_gemv_seq stores the launch's CUDA error in *cuda_err.
constexpr int kGemvSeqMaxJobs = 256;
int gemv_seq_workspace(const q4k_gemv_job* jobs, int n_jobs, int batch, size_t* bytes);
int launch_gemv_seq(const q4k_gemv_job* jobs, int n_jobs, int batch, void* workspace, size_t workspace_bytes,
                    cudaStream_t s, cudaError_t* cuda_err);
// Prepared job lists: the host plan (tensor maps, launch shapes, bound
// workspace) built once and launched many times.
size_t gemv_seq_plan_bytes(int n_jobs);
int gemv_seq_plan(const q4k_gemv_job* jobs, int n_jobs, int batch, void* workspace, size_t workspace_bytes,
                  void* plan, size_t plan_bytes, cudaError_t* cuda_err);
int gemv_seq_launch(const void* plan, cudaStream_t s, cudaError_t* cuda_err);
// Q4K_OK when `plan` is a valid plan made on the current device (enqueues nothing).
int gemv_seq_check_plan(const void* plan, cudaError_t* cuda_err);
// The same with the library's built-in scratch array as the workspace.
int launch_gemv_seq_static(const q4k_gemv_job* jobs, int n_jobs, int batch, cudaStream_t s,
                           cudaError_t* cuda_err);

// Tensor-core prefill MMQ GEMM (tcgen05).  When `p_out` is non-null the
// kernel stores the raw per-block integer dots there instead of y (test
// export); `err` is the device error word a timed-out wait sets.
bool gemm_tc_supported(int64_t tokens);
cudaError_t launch_gemm_block144(const uint8_t* w, int64_t rows, int64_t cols,
                                 const int8_t* q8, const float* d8,
                                 const int32_t* sum, int64_t tokens, float* y,
                                 int32_t* p_out, int* err, cudaStream_t s);

// Tensor-core prefill MMQ GEMM over binary16 quants (tensor copies load the
// activation operand directly).  p_out as for launch_gemm_block144.
cudaError_t launch_gemm_h16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* q16, const float* d8,
                            const int32_t* sum, int64_t tokens, float* y, int32_t* p_out, int* err,
                            cudaStream_t s);

// fp16-activation prefill GEMM: x split into per-token-scaled hi/lo binary16
// parts and block sums (x_split_f16), then the tensor-core GEMM over them.
cudaError_t launch_x_split_f16(const float* x, int64_t tokens, int64_t cols, uint16_t* hi, uint16_t* lo,
                               uint16_t* bsum, float* inv_scale, cudaStream_t s);
cudaError_t launch_gemm_f16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                            const uint16_t* bsum, const float* inv_scale, int64_t tokens, float* y, int* err,
                            cudaStream_t s);
// The same form over GPU-layout Q6_K weights (no min term, no block sums).
cudaError_t launch_gemm_q6k_f16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                                const float* inv_scale, int64_t tokens, float* y, int* err, cudaStream_t s);

// One-thread kernel whose only (bounded) wait can never complete: after the
// library's wait limit it records a timeout in `err` and returns.
cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t s);

}  // namespace q4k
