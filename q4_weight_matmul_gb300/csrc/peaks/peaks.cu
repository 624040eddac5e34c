// libq4k_peaks.so: tensor-core rate probes that the benchmark uses as the
// denominators of the prefill GEMM's roofline.  Not part of the Q4_K path.
//
//  - the dense int8 rate of the warp-level MMA (mma.sync m16n8k32 s8, the
//    only int8 tensor-core instruction sm_103a offers), and
//  - the dense fp16 rate of tcgen05.mma kind::f16 (M=128, N=256, K=16, one
//    CTA per SM, operands in shared memory), the instruction the GEMM uses.
//
// Both run register- or shared-memory-resident loops long enough (tens of
// ms) to reach a steady rate, timed with CUDA events.
#include "../tc_ptx.cuh"

#include <cuda_runtime.h>
#include <cstdint>

namespace {

using namespace q4k;

__global__ void __launch_bounds__(256) mma_s8_loop(int iters, int* sink) {
  int a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 ^ 0x1234, b1 = a0 ^ 0x5678;
  int acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  if (s == 0x7fffffff) sink[0] = s;   // keeps the loop alive
}

// One thread per CTA issues `groups` x 32 back-to-back M128 N256 K16 MMAs on
// zeroed shared-memory operands, at most two groups in flight.
__global__ void __launch_bounds__(128) tc_f16_loop(int groups, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc::fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tc::tmem_alloc(&tbase, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0) {
    const uint32_t id = tc::idesc_f16(128, 256, false);
    const uint32_t ab = tc::smem_u32(sm), bb = ab + 16384;
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ad[k] = tc::desc_sw128(ab + 32u * k);
      bd[k] = tc::desc_sw128(bb + 32u * k);
    }
    uint32_t phase = 0;
    bool ok = true;
    for (int g = 0; g < groups && ok; ++g) {
#pragma unroll
      for (int i = 0; i < 32; ++i) tc::mma_f16_ss(tbase, ad[i & 3], bd[i & 3], id, (g | i) ? 1u : 0u);
      tc::mma_commit(&bar);
      if (g >= 1) {
        ok = tc::mbar_wait_sleep(&bar, phase);
        phase ^= 1;
      }
    }
    if (ok) ok = tc::mbar_wait_sleep(&bar, phase);
    if (!ok) atomicOr(err, 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, 256);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

extern "C" {

// Dense int8 tensor rate (TOPS, a multiply-add counts 2) of mma.sync
// m16n8k32 s8 over `iters` iterations of 8 independent MMAs per warp, 4 CTAs
// of 256 threads per SM.  Returns 0, or a cudaError_t value.
int q4kp_mma_s8_tops(int iters, double* tops) {
  int* sink = nullptr;
  cudaError_t e = cudaMalloc(&sink, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  const int grid = 4 * sm_count();
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  mma_s8_loop<<<grid, 256>>>(64, sink);
  cudaEventRecord(e0);
  mma_s8_loop<<<grid, 256>>>(iters, sink);
  cudaEventRecord(e1);
  e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  *tops = 2.0 * 16 * 8 * 32 * 8.0 * iters * (grid * 8.0) / (ms * 1e-3) / 1e12;
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(sink);
  return (int)e;
}

// Dense fp16 tensor rate (TFLOP/s) of tcgen05.mma kind::f16, M=128 N=256
// K=16, one CTA per SM, `groups` x 32 MMAs per CTA.  Returns 0, a
// cudaError_t value, or -1 if a bounded wait gave up.
int q4kp_tc_f16_tflops(int groups, double* tflops) {
  int* err = nullptr;
  cudaError_t e = cudaMalloc(&err, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  cudaMemset(err, 0, sizeof(int));
  const int smem = 50 * 1024, grid = sm_count();
  e = cudaFuncSetAttribute(tc_f16_loop, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    cudaFree(err);
    return (int)e;
  }
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  tc_f16_loop<<<grid, 128, smem>>>(4, err);
  cudaEventRecord(e0);
  tc_f16_loop<<<grid, 128, smem>>>(groups, err);
  cudaEventRecord(e1);
  e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  int h = 0;
  cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
  *tflops = 2.0 * 128 * 256 * 16 * 32.0 * groups * grid / (ms * 1e-3) / 1e12;
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(err);
  return e != cudaSuccess ? (int)e : (h ? -1 : 0);
}

}  // extern "C"
