// q4k_gemv: decode GEMV y[b][o] = sum_k w[o][k] x[b][k] (+ residual) over
// BLOCK144 Q4_K weights (genie-ai-runtime §4, Path C: packed quants read as
// whole words, dequantised in registers, residual folded in).
//
// Mapping.  One CTA of 1024 threads per SM (persistent).  A warp owns 8 rows;
// lane (r, c) = (lane/4, lane%4) handles row r and the 64-weight chunk c of
// every superblock it visits: its 32 quant bytes hold all of sub-block 2c
// (low nibbles) and sub-block 2c+1 (high nibbles).  Warps split K when there
// are too few rows to fill the machine (KS warps per 8-row group, summed in
// shared memory in a fixed order, so results are bitwise deterministic).
//
// Dequantisation cost.  A nibble at bit position p (p <= 16) ORed into the
// float 2^23 gives 2^23 + q*2^p exactly; subtracting 2^23 leaves q*2^p, and
// the activation staged for that position is pre-multiplied by 2^-p, so the
// product is exactly q*x before its usual fp32 rounding.  Eight nibbles of a
// word need one shift, eight LOP3s, four packed fp32x2 adds and four packed
// fp32x2 FMAs per token.  Each sub-block's partial sum is then scaled:
//   acc += d*(sc_lo*S_lo + sc_hi*S_hi) - dmin*(m_lo*X_lo + m_hi*X_hi)
// where X_j = sum of x over sub-block j (staged once per CTA).
#include "q4k_internal.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kRegion = 68;   // floats per (token, superblock, chunk): 32 (lo,hi) pairs + pad

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float magic(uint32_t bits) { return __uint_as_float(0x4B000000u | bits); }

// Power-of-two pre-scale exponent of weight l (0..31) of the low (hi = 0) or
// high (hi = 1) half of a chunk; matches the nibble positions used below.
__device__ __forceinline__ int nib_shift(int l, int hi) {
  const uint32_t lo_tab = 0u | (8u << 8) | (16u << 16) | (12u << 24);
  const uint32_t hi_tab = 4u | (12u << 8) | (8u << 16) | (16u << 24);
  return (int)(((hi ? hi_tab : lo_tab) >> (8 * (l & 3))) & 0xFFu);
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_block144_kernel(
    const uint4* __restrict__ w, int rows, int nb, int ks,
    const float* __restrict__ x, const float* __restrict__ residual,
    float* __restrict__ y) {
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                                  // [B][nb][4][kRegion]
  float* xsum = xs + (size_t)B * nb * 4 * kRegion;   // [B][nb*8]
  float* red = xsum + (size_t)B * nb * 8;            // [kWarps][8][B]
  const int cols = nb * kQK;
  const int tid = threadIdx.x;

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Stage the activations: pre-scaled by 2^-p and paired (lo, hi) per chunk.
  for (int i = tid; i < B * cols; i += kThreads) {
    const int b = i / cols, k = i - b * cols;
    const int s = k >> 8, r = k & 255, c = r >> 6, t = r & 63;
    const int hi = t >> 5, l = t & 31;
    const float scale = __uint_as_float((uint32_t)(127 - nib_shift(l, hi)) << 23);
    xs[(((size_t)b * nb + s) * 4 + c) * kRegion + 2 * l + hi] = x[(size_t)b * cols + k] * scale;
  }
  for (int i = tid; i < B * nb * 8; i += kThreads) {
    const int b = i / (nb * 8), j = i - b * nb * 8;
    const float* xp = x + (size_t)b * cols + 32 * j;
    float acc = 0.0f;
    for (int t = 0; t < 32; ++t) acc += xp[t];
    xsum[i] = acc;
  }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  const int r8 = lane >> 2, c = lane & 3;
  const int groups_per_cta = kWarps / ks;
  const int g = warp / ks, z = warp - g * ks;
  const int n_groups = (rows + 7) >> 3;
  const int sh = (c & 1) * 16;
  const float2 kMagic2 = make_float2(-8388608.0f, -8388608.0f);

  for (int base = blockIdx.x * groups_per_cta; base < n_groups; base += gridDim.x * groups_per_cta) {
    const int grp = base + g;
    const int row = grp * 8 + r8;
    const bool valid = (grp < n_groups) && (row < rows);
    const uint4* wrow = w + (size_t)(valid ? row : 0) * nb * 9;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;

    uint4 hd = make_uint4(0, 0, 0, 0), q0 = hd, q1 = hd;
    if (valid && z < nb) {
      hd = ld_stream(wrow + z * 9);
      q0 = ld_stream(wrow + z * 9 + 1 + 2 * c);
      q1 = ld_stream(wrow + z * 9 + 2 + 2 * c);
    }
    for (int s = z; s < nb; s += ks) {
      uint4 hdn = make_uint4(0, 0, 0, 0), q0n = hdn, q1n = hdn;
      if (valid && s + ks < nb) {
        const uint4* p = wrow + (s + ks) * 9;
        hdn = ld_stream(p);
        q0n = ld_stream(p + 1 + 2 * c);
        q1n = ld_stream(p + 2 + 2 * c);
      }
      // scales and mins of sub-blocks 2c (lo) and 2c+1 (hi)
      const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
      const uint32_t a1 = hd.y >> sh, a2 = hd.z >> sh, a3 = hd.w >> sh;
      uint32_t sc01, m01;
      if (c < 2) {
        sc01 = a1 & 0x3F3Fu;
        m01 = a2 & 0x3F3Fu;
      } else {
        sc01 = (a3 & 0x0F0Fu) | ((a1 >> 2) & 0x3030u);
        m01 = ((a3 >> 4) & 0x0F0Fu) | ((a2 >> 2) & 0x3030u);
      }
      const float sc_lo = (float)(sc01 & 0xFFu), sc_hi = (float)(sc01 >> 8);
      const float m_lo = (float)(m01 & 0xFFu), m_hi = (float)(m01 >> 8);

      float2 part[B];
#pragma unroll
      for (int b = 0; b < B; ++b) part[b] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 qq = h ? q1 : q0;
        const uint32_t words[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t v = words[k], v12 = v >> 12;
          const float2 f0 = __fadd2_rn(make_float2(magic(v & 0xFu), magic(v & 0xF0u)), kMagic2);
          const float2 f1 = __fadd2_rn(make_float2(magic(v & 0xF00u), magic(v & 0xF000u)), kMagic2);
          const float2 f2 = __fadd2_rn(make_float2(magic(v & 0xF0000u), magic(v12 & 0xF00u)), kMagic2);
          const float2 f3 = __fadd2_rn(make_float2(magic(v12 & 0xF000u), magic(v12 & 0xF0000u)), kMagic2);
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const float4* xp = reinterpret_cast<const float4*>(
                xs + (((size_t)b * nb + s) * 4 + c) * kRegion + 2 * (16 * h + 4 * k));
            const float4 xa = xp[0], xb = xp[1];
            part[b] = __ffma2_rn(f0, make_float2(xa.x, xa.y), part[b]);
            part[b] = __ffma2_rn(f1, make_float2(xa.z, xa.w), part[b]);
            part[b] = __ffma2_rn(f2, make_float2(xb.x, xb.y), part[b]);
            part[b] = __ffma2_rn(f3, make_float2(xb.z, xb.w), part[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float2 xsm = *reinterpret_cast<const float2*>(xsum + (size_t)b * nb * 8 + s * 8 + 2 * c);
        const float scaled = fmaf(sc_hi, part[b].y, sc_lo * part[b].x);
        const float mins = fmaf(m_hi, xsm.y, m_lo * xsm.x);
        acc[b] = fmaf(dm.x, scaled, acc[b]);
        acc[b] = fmaf(-dm.y, mins, acc[b]);
      }
      hd = hdn;
      q0 = q0n;
      q1 = q1n;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
    }
    if (ks == 1) {
      if (valid && c == 0) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
          float v = acc[b];
          if (residual) v += residual[(size_t)b * rows + row];
          y[(size_t)b * rows + row] = v;
        }
      }
    } else {
      if (c == 0) {
#pragma unroll
        for (int b = 0; b < B; ++b) red[(warp * 8 + r8) * B + b] = acc[b];
      }
      __syncthreads();
      if (z == 0 && c == 0 && valid) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
          float v = 0.0f;
          for (int zz = 0; zz < ks; ++zz) v += red[((warp + zz) * 8 + r8) * B + b];
          if (residual) v += residual[(size_t)b * rows + row];
          y[(size_t)b * rows + row] = v;
        }
      }
      __syncthreads();
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

size_t smem_bytes(int batch, int nb) {
  return sizeof(float) * ((size_t)batch * nb * (4 * kRegion + 8) + (size_t)kWarps * 8 * batch);
}

template <int B>
cudaError_t launch_b(const uint8_t* w, int rows, int nb, const float* x,
                     const float* residual, float* y, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo& info = device_info(dev);
  const size_t smem = smem_bytes(B, nb);
  // raise the kernel's dynamic shared-memory limit once per device (it only grows)
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if ((int)smem > limit) {
    cudaError_t e = cudaFuncSetAttribute(gemv_block144_kernel<B>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin);
    if (e != cudaSuccess) return e;
    limit = info.max_smem_optin;
  }
  const int n_groups = (rows + 7) / 8;
  // split K across warps until every SM has a full CTA of work
  int ks = 1;
  while (ks < 8 && ks * 2 <= nb && (int64_t)n_groups * ks < (int64_t)info.sm_count * kWarps) ks *= 2;
  const int groups_per_cta = kWarps / ks;
  int grid = (n_groups + groups_per_cta - 1) / groups_per_cta;
  if (grid > info.sm_count) grid = info.sm_count;
  gemv_block144_kernel<B><<<grid, kThreads, smem, s>>>(
      reinterpret_cast<const uint4*>(w), rows, nb, ks, x, residual, y);
  return cudaGetLastError();
}

}  // namespace

bool gemv_supported(int64_t cols, int batch) {
  if (batch < 1 || batch > 8) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return smem_bytes(batch, (int)(cols / kQK)) <= (size_t)device_info(dev).max_smem_optin;
}

cudaError_t launch_gemv_block144(const uint8_t* w, int64_t rows, int64_t cols,
                                 const float* x, int batch,
                                 const float* residual, float* y,
                                 cudaStream_t s) {
  if (rows == 0 || batch == 0) return cudaSuccess;
  const int nb = (int)(cols / kQK);
  switch (batch) {
    case 1: return launch_b<1>(w, (int)rows, nb, x, residual, y, s);
    case 2: return launch_b<2>(w, (int)rows, nb, x, residual, y, s);
    case 3: return launch_b<3>(w, (int)rows, nb, x, residual, y, s);
    case 4: return launch_b<4>(w, (int)rows, nb, x, residual, y, s);
    case 5: return launch_b<5>(w, (int)rows, nb, x, residual, y, s);
    case 6: return launch_b<6>(w, (int)rows, nb, x, residual, y, s);
    case 7: return launch_b<7>(w, (int)rows, nb, x, residual, y, s);
    case 8: return launch_b<8>(w, (int)rows, nb, x, residual, y, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace q4k
