// q8_quantize: fp32 activations -> q8_1 blocks of 32 (int8 quants, an fp32
// scale and the block sum); q8_quantize_h16 stores the same quants as exact
// binary16 integers, the operand form the tensor-core GEMM loads directly.  Eight lanes share one block (four floats each):
// a 3-step shuffle gives the block's max |x| and its quant sum.  IEEE
// division (__fdiv_rn) and roundf (ties away from zero) make the result
// bit-reproducible against any correctly rounded implementation.
#include "q4k_internal.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

__device__ __forceinline__ int quant1(float v, float dd) {
  float r = roundf(__fdiv_rn(v, dd));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return (int)r;
}

__device__ __forceinline__ void store_q(char4* q, int64_t v, int a, int b, int c, int d) {
  q[v] = make_char4((signed char)a, (signed char)b, (signed char)c, (signed char)d);
}
// four binary16 integers (exact: |q| <= 127)
__device__ __forceinline__ void store_q(uint2* q, int64_t v, int a, int b, int c, int d) {
  const __half2 lo = __halves2half2(__int2half_rn(a), __int2half_rn(b));
  const __half2 hi = __halves2half2(__int2half_rn(c), __int2half_rn(d));
  q[v] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

template <typename QT>
__global__ void __launch_bounds__(256) q8_quantize_kernel(
    const float4* __restrict__ x, int64_t n_vec, QT* __restrict__ q,
    float* __restrict__ d8, int32_t* __restrict__ sum) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
    const float4 a = x[v];
    float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float dd = __fdiv_rn(amax, 127.0f);
    int qx = 0, qy = 0, qz = 0, qw = 0;
    if (dd != 0.0f) {
      qx = quant1(a.x, dd);
      qy = quant1(a.y, dd);
      qz = quant1(a.z, dd);
      qw = quant1(a.w, dd);
    }
    int s = qx + qy + qz + qw;
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    store_q(q, v, qx, qy, qz, qw);
    if ((threadIdx.x & 7) == 0) {
      d8[v >> 3] = dd;
      sum[v >> 3] = s;
    }
  }
}

}  // namespace

namespace {
int q8_grid(int64_t n_vec) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t want = (n_vec + 255) / 256;
  const int64_t cap = (int64_t)device_info(dev).sm_count * 8;
  return (int)(want < cap ? want : cap);
}
}  // namespace

cudaError_t launch_q8_quantize(const float* x, int64_t tokens, int64_t cols,
                               int8_t* q, float* d8, int32_t* sum,
                               cudaStream_t s) {
  const int64_t n_vec = tokens * cols / 4;   // a multiple of 64: whole warps
  if (n_vec == 0) return cudaSuccess;
  q8_quantize_kernel<char4><<<q8_grid(n_vec), 256, 0, s>>>(reinterpret_cast<const float4*>(x), n_vec,
                                                          reinterpret_cast<char4*>(q), d8, sum);
  return cudaGetLastError();
}

cudaError_t launch_q8_quantize_h16(const float* x, int64_t tokens, int64_t cols, uint16_t* q, float* d8,
                                   int32_t* sum, cudaStream_t s) {
  const int64_t n_vec = tokens * cols / 4;
  if (n_vec == 0) return cudaSuccess;
  q8_quantize_kernel<uint2><<<q8_grid(n_vec), 256, 0, s>>>(reinterpret_cast<const float4*>(x), n_vec,
                                                          reinterpret_cast<uint2*>(q), d8, sum);
  return cudaGetLastError();
}

}  // namespace q4k
