// The C ABI of libq4k.so (declared in include/q4k.h): host-side argument
// validation, then one asynchronous launch on the caller's stream.  Nothing
// here allocates device memory; the only device state the library owns is a
// per-device error word that kernels with bounded waits set when they give up.
#include "q4k_internal.h"
#include "tmap.h"

#include <cudaTypedefs.h>
#include <q4k.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace q4k {

__device__ int g_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices];
int* g_error_ptr[kMaxDevices];
thread_local char g_last_error[256] = "";

int record_cuda(cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return Q4K_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cols(int64_t cols) {
  if (cols <= 0 || cols % kQK != 0 || cols > (int64_t(1) << 24)) return Q4K_ERR_INVALID_ARG;
  return Q4K_OK;
}

int check_layout(int layout) {
  return layout == Q4K_LAYOUT_BLOCK144 ? Q4K_OK : Q4K_ERR_UNSUPPORTED;
}

int check_rows(int64_t rows) {
  return (rows < 0 || rows > (int64_t(1) << 24)) ? Q4K_ERR_INVALID_ARG : Q4K_OK;
}

}  // namespace

const DeviceInfo& device_info(int device) {
  if (device < 0 || device >= kMaxDevices) device = 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_info_ready[device]) {
    DeviceInfo& d = g_info[device];
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, device);
    if (d.sm_count <= 0) d.sm_count = 1;
    g_info_ready[device] = true;
  }
  return g_info[device];
}

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_error_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_error_ptr[dev] = static_cast<int*>(p);
  }
  return g_error_ptr[dev];
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                    uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  const cuuint64_t gdim[2] = {dim0, dim1};
  const cuuint64_t gstride[1] = {row_stride_bytes};
  const cuuint32_t bdim[2] = {box0, box1};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(map, dtype, 2, const_cast<void*>(base), gdim, gstride, bdim, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_u8_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                       const uint64_t strides[2], const uint32_t box[3]) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t gstride[2] = {strides[0], strides[1]};
  const cuuint32_t bdim[3] = {box[0], box[1], box[2]};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gdim, gstride,
                      bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace q4k

using namespace q4k;

extern "C" {

size_t q4k_packed_bytes(int64_t rows, int64_t cols, int layout) {
  if (check_rows(rows) || check_cols(cols) || check_layout(layout)) return 0;
  return (size_t)rows * (size_t)(cols / kQK) * kBlockBytes;
}

int q4k_pack(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc,
             const uint8_t* m, const uint8_t* q, int64_t rows, int64_t cols,
             int layout, void* w, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (rows == 0) return Q4K_OK;
  if (!d || !dmin || !sc || !m || !q || !w) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(d) || !aligned16(dmin) || !aligned16(sc) || !aligned16(m) || !aligned16(q) ||
      !aligned16(w))
    return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_pack_block144(d, dmin, sc, m, q, rows, cols, static_cast<uint8_t*>(w),
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

size_t q8_1_bytes(int64_t tokens, int64_t cols) {
  if (tokens < 0 || tokens > (int64_t(1) << 24) || check_cols(cols)) return 0;
  return (size_t)tokens * (size_t)cols + 2 * sizeof(int32_t) * (size_t)tokens * (size_t)(cols / kSub);
}

int q4k_unpack(const void* w, int layout, int64_t rows, int64_t cols, uint16_t* d, uint16_t* dmin,
               uint8_t* sc, uint8_t* m, uint8_t* q, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (rows == 0) return Q4K_OK;
  if (!w || !d || !dmin || !sc || !m || !q) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(d) || !aligned16(dmin) || !aligned16(sc) || !aligned16(m) || !aligned16(q))
    return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_unpack_block144(static_cast<const uint8_t*>(w), rows, cols, d, dmin, sc, m, q,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q8_quantize(const float* x, int64_t tokens, int64_t cols, int8_t* q, float* d8,
                int32_t* sum, void* stream) {
  if (tokens < 0 || tokens > (int64_t(1) << 24)) return Q4K_ERR_INVALID_ARG;
  if (int e = check_cols(cols)) return e;
  if (tokens == 0) return Q4K_OK;
  if (!x || !q || !d8 || !sum) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d8) || !aligned16(sum)) return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_q8_quantize(x, tokens, cols, q, d8, sum, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q8_quantize_h16(const float* x, int64_t tokens, int64_t cols, uint16_t* q, float* d8, int32_t* sum,
                    void* stream) {
  if (tokens < 0 || tokens > (int64_t(1) << 24)) return Q4K_ERR_INVALID_ARG;
  if (int e = check_cols(cols)) return e;
  if (tokens == 0) return Q4K_OK;
  if (!x || !q || !d8 || !sum) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d8) || !aligned16(sum)) return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_q8_quantize_h16(x, tokens, cols, q, d8, sum, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemv_multi(int n, const void* const* w, int layout, const int64_t* rows, int64_t cols,
                   const float* x, int64_t batch, const float* const* residual, float* const* y,
                   void* stream) {
  if (n < 1 || n > gemv_max_mats()) return n < 1 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  if (!w || !rows || !y) return Q4K_ERR_INVALID_ARG;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (batch < 0 || batch > 8) return batch < 0 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  // drop empty matrices; nothing to do if all are empty
  const uint8_t* wk[8];
  int64_t rk[8];
  const float* resk[8];
  float* yk[8];
  int k = 0;
  for (int m = 0; m < n; ++m) {
    if (int e = check_rows(rows[m])) return e;
    if (rows[m] == 0) continue;
    if (!w[m] || !y[m]) return Q4K_ERR_INVALID_ARG;
    const float* r = residual ? residual[m] : nullptr;
    if (!aligned16(w[m]) || !aligned16(y[m]) || (r && !aligned16(r))) return Q4K_ERR_ALIGNMENT;
    wk[k] = static_cast<const uint8_t*>(w[m]);
    rk[k] = rows[m];
    resk[k] = r;
    yk[k] = y[m];
    ++k;
  }
  if (k == 0 || batch == 0) return Q4K_OK;
  if (!x) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(x)) return Q4K_ERR_ALIGNMENT;
  if (!gemv_supported(rk, k, cols, (int)batch)) return Q4K_ERR_UNSUPPORTED;
  cudaError_t e = launch_gemv_block144(wk, rk, k, cols, x, (int)batch, resk, yk,
                                       static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return Q4K_ERR_UNSUPPORTED;
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemv_q8(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8, const float* d8,
                const int32_t* sum, int64_t batch, const float* residual, float* y, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (batch < 0 || batch > 8) return batch < 0 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return Q4K_OK;
  if (!w || !q8 || !d8 || !sum || !y) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q8) || !aligned16(d8) || !aligned16(sum) || !aligned16(y) ||
      (residual && !aligned16(residual)))
    return Q4K_ERR_ALIGNMENT;
  if (!gemv_q8_supported(rows, cols, (int)batch)) return Q4K_ERR_UNSUPPORTED;
  cudaError_t e = launch_gemv_q8_block144(static_cast<const uint8_t*>(w), rows, cols, q8, false, d8, sum,
                                          (int)batch, residual, y, nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemv(const void* w, int layout, int64_t rows, int64_t cols, const float* x,
             int64_t batch, const float* residual, float* y, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (batch < 0 || batch > 8) return batch < 0 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return Q4K_OK;
  if (!w || !x || !y) return Q4K_ERR_INVALID_ARG;
  const float* const res[1] = {residual};
  float* const ys[1] = {y};
  return q4k_gemv_multi(1, &w, layout, &rows, cols, x, batch, res, ys, stream);
}

static bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

static int check_q6_layout(int layout) {
  return (layout == Q6K_LAYOUT_GGUF || layout == Q6K_LAYOUT_GPU) ? Q4K_OK : Q4K_ERR_UNSUPPORTED;
}

size_t q6k_packed_bytes(int64_t rows, int64_t cols, int layout) {
  if (check_rows(rows) || check_cols(cols) || check_q6_layout(layout)) return 0;
  const int64_t nb = cols / kQK;
  return layout == Q6K_LAYOUT_GGUF ? (size_t)rows * (size_t)nb * kQ6GgufBytes
                                   : (size_t)rows * (size_t)q6k_gpu_row_bytes(nb);
}

// a packed buffer's alignment: 2 bytes for GGUF blocks, 16 for the GPU layout
static bool q6_aligned(const void* w, int layout) {
  return layout == Q6K_LAYOUT_GGUF ? aligned2(w) : aligned16(w);
}

int q6k_pack(const uint16_t* d, const int8_t* sc, const uint8_t* q, int64_t rows, int64_t cols, int layout,
             void* w, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_q6_layout(layout)) return e;
  if (rows == 0) return Q4K_OK;
  if (!d || !sc || !q || !w) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(d) || !aligned16(sc) || !aligned16(q) || !aligned16(w)) return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_q6k_convert(d, sc, q, nullptr, -1, rows, cols, nullptr, nullptr, nullptr,
                                     static_cast<uint8_t*>(w), layout, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q6k_repack(const void* src, int src_layout, int64_t rows, int64_t cols, void* dst, int dst_layout,
               void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_q6_layout(src_layout)) return e;
  if (int e = check_q6_layout(dst_layout)) return e;
  if (rows == 0) return Q4K_OK;
  if (!src || !dst) return Q4K_ERR_INVALID_ARG;
  if (!q6_aligned(src, src_layout) || !q6_aligned(dst, dst_layout)) return Q4K_ERR_ALIGNMENT;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const size_t sn = q6k_packed_bytes(rows, cols, src_layout), dn = q6k_packed_bytes(rows, cols, dst_layout);
  if (s0 < d0 + dn && d0 < s0 + sn) return Q4K_ERR_INVALID_ARG;   // overlap
  cudaError_t e = launch_q6k_convert(nullptr, nullptr, nullptr, static_cast<const uint8_t*>(src), src_layout, rows,
                                     cols, nullptr, nullptr, nullptr, static_cast<uint8_t*>(dst), dst_layout,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q6k_unpack(const void* w, int layout, int64_t rows, int64_t cols, uint16_t* d, int8_t* sc, uint8_t* q,
               void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_q6_layout(layout)) return e;
  if (rows == 0) return Q4K_OK;
  if (!w || !d || !sc || !q) return Q4K_ERR_INVALID_ARG;
  if (!q6_aligned(w, layout) || !aligned16(d) || !aligned16(sc) || !aligned16(q)) return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_q6k_convert(nullptr, nullptr, nullptr, static_cast<const uint8_t*>(w), layout, rows, cols,
                                     d, sc, q, nullptr, -1, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q6k_gemv(const void* w, int layout, int64_t rows, int64_t cols, const float* x, int64_t batch,
             const float* residual, float* y, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_q6_layout(layout)) return e;
  if (batch < 0) return Q4K_ERR_INVALID_ARG;
  if (layout != Q6K_LAYOUT_GPU || batch > 8) return Q4K_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return Q4K_OK;
  if (!w || !x || !y) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)))
    return Q4K_ERR_ALIGNMENT;
  if (!gemv_q6k_supported(rows, cols, (int)batch)) return Q4K_ERR_UNSUPPORTED;
  cudaError_t e = launch_gemv_q6k(static_cast<const uint8_t*>(w), rows, cols, x, (int)batch, residual, y,
                                  static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return Q4K_ERR_UNSUPPORTED;
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

// shape and layout checks of the Q6_K q8_1 products (the GPU layout only)
static int check_q6k_mmq(int layout, int64_t rows, int64_t cols) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_q6_layout(layout)) return e;
  return layout == Q6K_LAYOUT_GPU ? Q4K_OK : Q4K_ERR_UNSUPPORTED;
}

int q6k_gemv_q8(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8, const float* d8,
                const int32_t* sum, int64_t batch, const float* residual, float* y, void* stream) {
  if (int e = check_q6k_mmq(layout, rows, cols)) return e;
  if (batch < 0 || batch > 8) return batch < 0 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return Q4K_OK;
  if (!w || !q8 || !d8 || !y) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q8) || !aligned16(d8) || (sum && !aligned16(sum)) || !aligned16(y) ||
      (residual && !aligned16(residual)))
    return Q4K_ERR_ALIGNMENT;
  if (!gemv_q6k_q8_supported(rows, cols, (int)batch)) return Q4K_ERR_UNSUPPORTED;
  cudaError_t e = launch_gemv_q6k_q8(static_cast<const uint8_t*>(w), rows, cols, q8, false, d8, nullptr, (int)batch,
                                     residual, y, nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

// q6k_gemm / q6k_gemm_blockdots: the MMQ product for any token count as
// q8_1 GEMV launches of up to 8 tokens each
static int q6k_gemm_common(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8, const float* d8,
                           int64_t tokens, float* y, int32_t* p, void* stream) {
  if (int e = check_q6k_mmq(layout, rows, cols)) return e;
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (rows == 0 || tokens == 0) return Q4K_OK;
  if (!w || !q8 || (!p && (!d8 || !y))) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q8) || (d8 && !aligned16(d8)) || (y && !aligned16(y)) || (p && !aligned16(p)))
    return Q4K_ERR_ALIGNMENT;
  // every launch's shape is checked before the first is enqueued
  const int64_t nsub = cols / kSub, ngrp = cols / 16;
  if (!gemv_q6k_q8_supported(rows, cols, (int)std::min<int64_t>(tokens, 8)) ||
      (tokens % 8 && !gemv_q6k_q8_supported(rows, cols, (int)(tokens % 8))))
    return Q4K_ERR_UNSUPPORTED;
  for (int64_t t0 = 0; t0 < tokens; t0 += 8) {
    const int n = (int)std::min<int64_t>(8, tokens - t0);
    cudaError_t e = launch_gemv_q6k_q8(static_cast<const uint8_t*>(w), rows, cols, q8 + t0 * cols, false,
                                       d8 ? d8 + t0 * nsub : nullptr, nullptr, n, nullptr, y ? y + t0 * rows : nullptr,
                                       p ? p + t0 * rows * ngrp : nullptr, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return record_cuda(e);
  }
  return Q4K_OK;
}

int q6k_gemm(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8, const float* d8,
             const int32_t* sum, int64_t tokens, float* y, void* stream) {
  (void)sum;   // the Q6_K product has no min term: the block sums are not read
  return q6k_gemm_common(w, layout, rows, cols, q8, d8, tokens, y, nullptr, stream);
}

int q6k_gemm_f16(const void* w, int layout, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                 const uint16_t* bsum, const float* inv_scale, int64_t tokens, float* y, void* stream) {
  (void)bsum;   // the Q6_K product has no min term: the block sums are not read
  if (int e = check_q6k_mmq(layout, rows, cols)) return e;
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (rows == 0 || tokens == 0) return Q4K_OK;
  if (!w || !hi || !lo || !inv_scale || !y) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(hi) || !aligned16(lo) || !aligned16(inv_scale) || !aligned16(y))
    return Q4K_ERR_ALIGNMENT;
  int* err = device_error_word();
  if (!err) return record_cuda(cudaGetLastError());
  cudaError_t e = launch_gemm_q6k_f16(static_cast<const uint8_t*>(w), rows, cols, hi, lo, inv_scale, tokens, y, err,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q6k_gemm_blockdots(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8, int64_t tokens,
                       int32_t* p, void* stream) {
  if (!p && rows != 0 && tokens != 0) return Q4K_ERR_INVALID_ARG;
  return q6k_gemm_common(w, layout, rows, cols, q8, nullptr, tokens, nullptr, p, stream);
}

// Host-side checks of a q4k_gemv_seq request (no CUDA call).  Sets *work to
// whether any job has work.
static int check_seq(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch, bool* work) {
  *work = false;
  if (n_jobs < 0) return Q4K_ERR_INVALID_ARG;
  if (n_jobs > kGemvSeqMaxJobs) return Q4K_ERR_UNSUPPORTED;
  if (n_jobs > 0 && !jobs) return Q4K_ERR_INVALID_ARG;
  if (int e = check_layout(layout)) return e;
  if (batch < 0 || batch > 8) return batch < 0 ? Q4K_ERR_INVALID_ARG : Q4K_ERR_UNSUPPORTED;
  for (int i = 0; i < n_jobs; ++i) {
    const q4k_gemv_job& j = jobs[i];
    if (int e = check_rows(j.rows)) return e;
    if (int e = check_cols(j.cols)) return e;
    if (j.format != 0 && j.format != 1) return Q4K_ERR_INVALID_ARG;
    if (j.rows == 0) continue;
    if (!j.w || !j.x || !j.y) return Q4K_ERR_INVALID_ARG;
    if (!aligned16(j.w) || !aligned16(j.x) || !aligned16(j.y) || (j.residual && !aligned16(j.residual)))
      return Q4K_ERR_ALIGNMENT;
    *work = true;
  }
  if (batch == 0) *work = false;
  return Q4K_OK;
}

// Token counts up to this go through the q8_1 GEMV (one weight pass per 8
// tokens) instead of a 128-token tensor-core tile.
constexpr int64_t kGemvTokens = 32;

// The MMQ product for a few tokens: q8_1 GEMV launches of up to 8 tokens.
static cudaError_t gemm_by_gemv(const uint8_t* w, int64_t rows, int64_t cols, const void* q8, bool h16,
                                const float* d8, const int32_t* sum, int64_t tokens, float* y, int32_t* p,
                                cudaStream_t s) {
  const int64_t nsub = cols / kSub;
  for (int64_t t0 = 0; t0 < tokens; t0 += 8) {
    const int n = (int)std::min<int64_t>(8, tokens - t0);
    const void* qt = h16 ? static_cast<const void*>(static_cast<const uint16_t*>(q8) + t0 * cols)
                         : static_cast<const void*>(static_cast<const int8_t*>(q8) + t0 * cols);
    cudaError_t e = launch_gemv_q8_block144(w, rows, cols, qt, h16, d8 ? d8 + t0 * nsub : nullptr,
                                            sum ? sum + t0 * nsub : nullptr, n, nullptr,
                                            y ? y + t0 * rows : nullptr, p ? p + t0 * rows * nsub : nullptr, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

static int gemm_common(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8,
                       const float* d8, const int32_t* sum, int64_t tokens, float* y,
                       int32_t* p, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (rows == 0 || tokens == 0) return Q4K_OK;
  if (!w || !q8) return Q4K_ERR_INVALID_ARG;
  if (!p && (!d8 || !sum || !y)) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q8) || (d8 && !aligned16(d8)) || (sum && !aligned16(sum)) ||
      (y && !aligned16(y)) || (p && !aligned16(p)))
    return Q4K_ERR_ALIGNMENT;
  cudaError_t e;
  if (tokens <= kGemvTokens) {
    if (!gemv_q8_supported(rows, cols, (int)std::min<int64_t>(tokens, 8))) return Q4K_ERR_UNSUPPORTED;
    e = gemm_by_gemv(static_cast<const uint8_t*>(w), rows, cols, q8, false, d8, sum, tokens, y, p,
                     static_cast<cudaStream_t>(stream));
  } else {
    int* err = device_error_word();
    if (!err) return record_cuda(cudaGetLastError());
    e = launch_gemm_block144(static_cast<const uint8_t*>(w), rows, cols, q8, d8, sum, tokens, y, p,
                             err, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemm(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8,
             const float* d8, const int32_t* sum, int64_t tokens, float* y, void* stream) {
  return gemm_common(w, layout, rows, cols, q8, d8, sum, tokens, y, nullptr, stream);
}

int q4k_gemm_blockdots(const void* w, int layout, int64_t rows, int64_t cols, const int8_t* q8,
                       int64_t tokens, int32_t* p, void* stream) {
  if (!p && rows != 0 && tokens != 0) return Q4K_ERR_INVALID_ARG;
  return gemm_common(w, layout, rows, cols, q8, nullptr, nullptr, tokens, nullptr, p, stream);
}

static int gemm_h16_common(const void* w, int layout, int64_t rows, int64_t cols, const uint16_t* q16,
                           const float* d8, const int32_t* sum, int64_t tokens, float* y, int32_t* p,
                           void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (rows == 0 || tokens == 0) return Q4K_OK;
  if (!w || !q16) return Q4K_ERR_INVALID_ARG;
  if (!p && (!d8 || !sum || !y)) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q16) || (d8 && !aligned16(d8)) || (sum && !aligned16(sum)) ||
      (y && !aligned16(y)) || (p && !aligned16(p)))
    return Q4K_ERR_ALIGNMENT;
  cudaError_t e;
  if (tokens <= kGemvTokens) {
    if (!gemv_q8_supported(rows, cols, (int)std::min<int64_t>(tokens, 8))) return Q4K_ERR_UNSUPPORTED;
    e = gemm_by_gemv(static_cast<const uint8_t*>(w), rows, cols, q16, true, d8, sum, tokens, y, p,
                     static_cast<cudaStream_t>(stream));
  } else {
    int* err = device_error_word();
    if (!err) return record_cuda(cudaGetLastError());
    e = launch_gemm_h16(static_cast<const uint8_t*>(w), rows, cols, q16, d8, sum, tokens, y, p, err,
                        static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemm_h16(const void* w, int layout, int64_t rows, int64_t cols, const uint16_t* q16, const float* d8,
                 const int32_t* sum, int64_t tokens, float* y, void* stream) {
  return gemm_h16_common(w, layout, rows, cols, q16, d8, sum, tokens, y, nullptr, stream);
}

int q4k_gemm_blockdots_h16(const void* w, int layout, int64_t rows, int64_t cols, const uint16_t* q16,
                           int64_t tokens, int32_t* p, void* stream) {
  if (!p && rows != 0 && tokens != 0) return Q4K_ERR_INVALID_ARG;
  return gemm_h16_common(w, layout, rows, cols, q16, nullptr, nullptr, tokens, nullptr, p, stream);
}

size_t x_split_f16_bytes(int64_t tokens, int64_t cols) {
  if (tokens < 0 || tokens > (int64_t(1) << 22) || check_cols(cols)) return 0;
  return (size_t)tokens * ((size_t)cols * 4 + (size_t)(cols / kQK) * 32 + 4);
}

int x_split_f16(const float* x, int64_t tokens, int64_t cols, uint16_t* hi, uint16_t* lo, uint16_t* bsum,
                float* inv_scale, void* stream) {
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (int e = check_cols(cols)) return e;
  if (tokens == 0) return Q4K_OK;
  if (!x || !hi || !lo || !bsum || !inv_scale) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(hi) || !aligned16(lo) || !aligned16(bsum) || !aligned16(inv_scale))
    return Q4K_ERR_ALIGNMENT;
  cudaError_t e = launch_x_split_f16(x, tokens, cols, hi, lo, bsum, inv_scale, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_gemm_f16(const void* w, int layout, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                 const uint16_t* bsum, const float* inv_scale, int64_t tokens, float* y, void* stream) {
  if (int e = check_rows(rows)) return e;
  if (int e = check_cols(cols)) return e;
  if (int e = check_layout(layout)) return e;
  if (tokens < 0 || tokens > (int64_t(1) << 22)) return Q4K_ERR_INVALID_ARG;
  if (rows == 0 || tokens == 0) return Q4K_OK;
  if (!w || !hi || !lo || !bsum || !inv_scale || !y) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(hi) || !aligned16(lo) || !aligned16(bsum) || !aligned16(inv_scale) ||
      !aligned16(y))
    return Q4K_ERR_ALIGNMENT;
  int* err = device_error_word();
  if (!err) return record_cuda(cudaGetLastError());
  cudaError_t e = launch_gemm_f16(static_cast<const uint8_t*>(w), rows, cols, hi, lo, bsum, inv_scale, tokens, y,
                                  err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

size_t q4k_gemv_seq_workspace_bytes(const q4k_gemv_job* jobs, int n_jobs, int64_t batch) {
  bool work = false;
  if (check_seq(jobs, n_jobs, Q4K_LAYOUT_BLOCK144, batch, &work) != Q4K_OK || !work) return 0;
  size_t bytes = 0;
  if (gemv_seq_workspace(jobs, n_jobs, (int)batch, &bytes) != Q4K_OK) return 0;
  return bytes;
}

int q4k_gemv_seq(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch, void* workspace,
                 size_t workspace_bytes, void* stream) {
  bool work = false;
  if (int e = check_seq(jobs, n_jobs, layout, batch, &work)) return e;
  if (!work) return Q4K_OK;
  if (!workspace) return Q4K_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return Q4K_ERR_ALIGNMENT;
  cudaError_t ce = cudaSuccess;
  const int st = launch_gemv_seq(jobs, n_jobs, (int)batch, workspace, workspace_bytes,
                                 static_cast<cudaStream_t>(stream), &ce);
  if (st == Q4K_ERR_CUDA) return record_cuda(ce);
  return st;
}

size_t q4k_gemv_seq_plan_bytes(int n_jobs) {
  if (n_jobs < 0 || n_jobs > kGemvSeqMaxJobs) return 0;
  return gemv_seq_plan_bytes(n_jobs);
}

int q4k_gemv_seq_plan(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch, void* workspace,
                      size_t workspace_bytes, void* plan, size_t plan_bytes) {
  bool work = false;
  if (int e = check_seq(jobs, n_jobs, layout, batch, &work)) return e;
  if (!plan) return Q4K_ERR_INVALID_ARG;
  if (work) {
    if (!workspace) return Q4K_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return Q4K_ERR_ALIGNMENT;
  }
  cudaError_t ce = cudaSuccess;
  const int st = gemv_seq_plan(jobs, n_jobs, work ? (int)batch : 0, work ? workspace : nullptr,
                               workspace_bytes, plan, plan_bytes, &ce);
  if (st == Q4K_ERR_CUDA) return record_cuda(ce);
  return st;
}

int q4k_gemv_seq_launch(const void* plan, void* stream) {
  if (!plan) return Q4K_ERR_INVALID_ARG;
  cudaError_t ce = cudaSuccess;
  const int st = gemv_seq_launch(plan, static_cast<cudaStream_t>(stream), &ce);
  if (st == Q4K_ERR_CUDA) return record_cuda(ce);
  return st;
}

int q4k_gemv_seq_launch_host(const void* plan, const void* x_host, void* x_dev, size_t x_bytes, void* y_host,
                             const void* y_dev, size_t y_bytes, void* stream) {
  if (!plan) return Q4K_ERR_INVALID_ARG;
  if (x_bytes && (!x_host || !x_dev)) return Q4K_ERR_INVALID_ARG;
  if (y_bytes && (!y_host || !y_dev)) return Q4K_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaSuccess;
  if (const int st = gemv_seq_check_plan(plan, &ce)) return st == Q4K_ERR_CUDA ? record_cuda(ce) : st;
  if (x_bytes && (ce = cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return record_cuda(ce);
  const int st = gemv_seq_launch(plan, s, &ce);
  if (st == Q4K_ERR_CUDA) return record_cuda(ce);
  if (st != Q4K_OK) return st;
  if (y_bytes && (ce = cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return record_cuda(ce);
  return Q4K_OK;
}

int q4k_gemv_seq_static(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch, void* stream) {
  bool work = false;
  if (int e = check_seq(jobs, n_jobs, layout, batch, &work)) return e;
  if (!work) return Q4K_OK;
  cudaError_t ce = cudaSuccess;
  const int st = launch_gemv_seq_static(jobs, n_jobs, (int)batch, static_cast<cudaStream_t>(stream), &ce);
  if (st == Q4K_ERR_CUDA) return record_cuda(ce);
  return st;
}

int q4k_selftest_wait_timeout(void* stream) {
  int* err = device_error_word();
  if (!err) return record_cuda(cudaGetLastError());
  cudaError_t e = launch_wait_timeout_selftest(err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q4K_OK : record_cuda(e);
}

int q4k_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e);
  int* word = device_error_word();
  if (!word) return record_cuda(cudaGetLastError());
  int value = 0;
  e = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda(e);
  if (value != 0) {
    const int zero = 0;
    e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return record_cuda(e);
    return Q4K_ERR_DEVICE_TIMEOUT;
  }
  return Q4K_OK;
}

const char* q4k_status_string(int status) {
  switch (status) {
    case Q4K_OK: return "Q4K_OK";
    case Q4K_ERR_INVALID_ARG: return "Q4K_ERR_INVALID_ARG";
    case Q4K_ERR_ALIGNMENT: return "Q4K_ERR_ALIGNMENT";
    case Q4K_ERR_UNSUPPORTED: return "Q4K_ERR_UNSUPPORTED";
    case Q4K_ERR_CUDA: return "Q4K_ERR_CUDA";
    case Q4K_ERR_DEVICE_TIMEOUT: return "Q4K_ERR_DEVICE_TIMEOUT";
    default: return "Q4K_ERR_UNKNOWN";
  }
}

const char* q4k_last_error_string(void) { return g_last_error; }

const char* q4k_version(void) { return "q4k 0.1.0 sm_103a"; }

}  // extern "C"
