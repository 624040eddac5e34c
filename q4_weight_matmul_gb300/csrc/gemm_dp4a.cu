// Small-tile integer MMQ on CUDA cores (dp4a): the prefill GEMM for token
// counts too small to fill a tensor-core tile, and the independent GPU
// restatement of the per-block integer dots.
//
//   P[t][o][b] = sum_{i<32} q[o][32b+i] * q8[t][32b+i]          (exact int32)
//   y[t][o]    = sum_b d*sc[o,b] * d8[t,b] * P - dmin*m[o,b] * d8[t,b] * S[t,b]
//
// A CTA of 256 threads owns a 64-row x 64-token tile and walks K one
// superblock at a time: the 64 packed superblocks (9 KB) and the 64x256 q8
// tile (16 KB) are staged in shared memory, the eight (d*sc, dmin*m) pairs of
// each row are decoded once per superblock, and each thread accumulates a
// 4x4 sub-tile with dp4a (four 4-bit quants widened to bytes by one mask).
#include "q4k_internal.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kTile = 64;
constexpr int kQ8Stride = 272;   // padded q8 row: 2-way bank conflicts at most

__global__ void __launch_bounds__(256) gemm_dp4a_kernel(
    const uint8_t* __restrict__ w, int rows, int nb, const int8_t* __restrict__ q8,
    const float* __restrict__ d8, const int32_t* __restrict__ ssum, int tokens,
    float* __restrict__ y, int32_t* __restrict__ p_out) {
  __shared__ __align__(16) uint8_t s_w[kTile * kBlockBytes];
  __shared__ __align__(16) int8_t s_q8[kTile * kQ8Stride];
  __shared__ float s_dsc[kTile][8], s_dmm[kTile][8], s_d8[kTile][8];
  __shared__ int s_sum[kTile][8];

  const int tid = threadIdx.x;
  const int row0 = blockIdx.x * kTile, tok0 = blockIdx.y * kTile;
  const int cols = nb * kQK;
  const int tr = tid >> 4, tt = tid & 15;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int s = 0; s < nb; ++s) {
    // stage 64 superblocks (one per row) and 64 tokens x 256 quants
    for (int i = tid; i < kTile * 9; i += 256) {
      const int r = i / 9, v = i - r * 9;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (row0 + r < rows)
        val = reinterpret_cast<const uint4*>(w + ((size_t)(row0 + r) * nb + s) * kBlockBytes)[v];
      reinterpret_cast<uint4*>(s_w)[i] = val;
    }
    for (int i = tid; i < kTile * 16; i += 256) {
      const int t = i >> 4, v = i & 15;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (tok0 + t < tokens)
        val = reinterpret_cast<const uint4*>(q8 + (size_t)(tok0 + t) * cols + s * kQK)[v];
      *reinterpret_cast<uint4*>(s_q8 + t * kQ8Stride + 16 * v) = val;
    }
    if (!p_out) {   // scales are not passed (null) when only block dots are wanted
      for (int i = tid; i < kTile * 8; i += 256) {
        const int t = i >> 3, j = i & 7;
        const bool ok = tok0 + t < tokens;
        s_d8[t][j] = ok ? d8[(size_t)(tok0 + t) * (cols / kSub) + s * 8 + j] : 0.0f;
        s_sum[t][j] = ok ? ssum[(size_t)(tok0 + t) * (cols / kSub) + s * 8 + j] : 0;
      }
    }
    __syncthreads();
    for (int i = tid; i < kTile * 8; i += 256) {
      const int r = i >> 3, j = i & 7;
      const uint8_t* h = s_w + r * kBlockBytes;
      const float d = __half2float(*reinterpret_cast<const __half*>(h));
      const float dmin = __half2float(*reinterpret_cast<const __half*>(h + 2));
      const uint8_t* sc = h + 4;
      int scv, mv;
      if (j < 4) {
        scv = sc[j] & 63;
        mv = sc[j + 4] & 63;
      } else {
        scv = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
        mv = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
      }
      s_dsc[r][j] = d * (float)scv;
      s_dmm[r][j] = dmin * (float)mv;
    }
    __syncthreads();

    for (int jb = 0; jb < 8; ++jb) {
      const int c = jb >> 1, hi = jb & 1;
      int p[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[i][j] = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        int a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t word =
              *reinterpret_cast<const uint32_t*>(s_w + (tr + 16 * i) * kBlockBytes + 16 + 32 * c + 4 * u);
          a[i] = (int)(hi ? ((word >> 4) & 0x0F0F0F0Fu) : (word & 0x0F0F0F0Fu));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          b[j] = *reinterpret_cast<const int*>(s_q8 + (tt + 16 * j) * kQ8Stride + 32 * jb + 4 * u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) p[i][j] = __dp4a(a[i], b[j], p[i][j]);
      }
      if (p_out) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = row0 + tr + 16 * i, t = tok0 + tt + 16 * j;
            if (r < rows && t < tokens)
              p_out[((size_t)t * rows + r) * (cols / kSub) + s * 8 + jb] = p[i][j];
          }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float dsc = s_dsc[tr + 16 * i][jb], dmm = s_dmm[tr + 16 * i][jb];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float dd = s_d8[tt + 16 * j][jb];
            const float u = dd * (float)s_sum[tt + 16 * j][jb];
            acc[i][j] = fmaf(dsc * dd, (float)p[i][j], acc[i][j]);
            acc[i][j] = fmaf(-dmm, u, acc[i][j]);
          }
        }
      }
    }
    __syncthreads();
  }
  if (!p_out) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = row0 + tr + 16 * i, t = tok0 + tt + 16 * j;
        if (r < rows && t < tokens) y[(size_t)t * rows + r] = acc[i][j];
      }
  }
}

}  // namespace

cudaError_t launch_gemm_dp4a(const uint8_t* w, int64_t rows, int64_t cols,
                             const int8_t* q8, const float* d8,
                             const int32_t* sum, int64_t tokens, float* y,
                             int32_t* p_out, cudaStream_t s) {
  if (rows == 0 || tokens == 0) return cudaSuccess;
  dim3 grid((unsigned)((rows + kTile - 1) / kTile), (unsigned)((tokens + kTile - 1) / kTile));
  gemm_dp4a_kernel<<<grid, 256, 0, s>>>(w, (int)rows, (int)(cols / kQK), q8, d8, sum,
                                        (int)tokens, y, p_out);
  return cudaGetLastError();
}

}  // namespace q4k
