// q4k_gemv: decode GEMV y[b][o] = sum_k w[o][k] x[b][k] (+ residual) over
// BLOCK144 Q4_K weights (genie-ai-runtime §4, Path C: packed quants read as
// whole words, dequantised in registers, residual folded in).
//
// Streaming.  One persistent CTA of 16 warps per SM.  Each warp owns a ring
// of kRing shared-memory stages; one stage holds one superblock (144 bytes)
// of each of the warp's 8 rows, fetched by eight cp.async.bulk copies that
// complete on the stage's mbarrier.  The first copies are issued before the
// activations are staged, so the weight stream starts at launch; afterwards a
// stage is refilled as soon as the warp has consumed it.  Bytes in flight are
// then set by the ring depth, not by registers.
//
// Mapping.  Lane (r, c) = (lane/4, lane%4) works on row r and the 64-weight
// chunk c of each superblock: its 32 quant bytes hold all of sub-block 2c
// (low nibbles) and all of sub-block 2c+1 (high nibbles).  When there are too
// few 8-row groups to occupy every warp, ks warps split a group's superblocks
// and their partial sums are added in shared memory in a fixed order, so the
// result is bitwise deterministic.
//
// Dequantisation.  A nibble at bit position p (p <= 16) ORed into the float
// 2^23 gives 2^23 + q*2^p exactly; subtracting 2^23 leaves q*2^p, and the
// activation staged for that position is pre-multiplied by 2^-p, so the
// product is exactly q*x before its fp32 rounding.  A word of eight nibbles
// costs one shift, eight LOP3s, four fp32x2 adds and four fp32x2 FMAs per
// token.  Each sub-block's partial dot is then scaled:
//   acc += d*(sc_lo*S_lo + sc_hi*S_hi) - dmin*(m_lo*X_lo + m_hi*X_hi)
// with X_j the sum of x over sub-block j (staged once per CTA).
#include "q4k_internal.h"
#include "tc_ptx.cuh"

#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRegion = 68;          // floats per (token, superblock, chunk): 32 (lo,hi) pairs + pad
constexpr int kStageBytes = 8 * kBlockBytes;

__device__ __forceinline__ float magic(uint32_t bits) { return __uint_as_float(0x4B000000u | bits); }

// Power-of-two pre-scale exponent of weight l (0..31) of the low (hi = 0) or
// high (hi = 1) half of a chunk; matches the nibble positions used below.
__device__ __forceinline__ int nib_shift(int l, int hi) {
  const uint32_t lo_tab = 0u | (8u << 8) | (16u << 16) | (12u << 24);
  const uint32_t hi_tab = 4u | (12u << 8) | (8u << 16) | (16u << 24);
  return (int)(((hi ? hi_tab : lo_tab) >> (8 * (l & 3))) & 0xFFu);
}

struct Layout {
  int B, nb, ring;
  size_t xs, xsum, red, stages, bars, total;
};

__host__ __device__ inline Layout layout(int B, int nb, int ring) {
  Layout L;
  L.B = B;
  L.nb = nb;
  L.ring = ring;
  L.xs = 0;
  L.xsum = L.xs + sizeof(float) * (size_t)B * nb * 4 * kRegion;
  L.red = L.xsum + sizeof(float) * (size_t)B * nb * 8;
  L.stages = (L.red + sizeof(float) * (size_t)kWarps * 8 * B + 127) & ~size_t(127);
  L.bars = L.stages + (size_t)kWarps * ring * kStageBytes;
  L.total = L.bars + sizeof(uint64_t) * kWarps * ring;
  return L;
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_block144_kernel(
    const uint8_t* __restrict__ w, int rows, int nb, int ks, int ring,
    const float* __restrict__ x, const float* __restrict__ residual,
    float* __restrict__ y, int* __restrict__ err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout L = layout(B, nb, ring);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  float* red = reinterpret_cast<float*>(smem + L.red);
  const int cols = nb * kQK;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r8 = lane >> 2, c = lane & 3;
  const int gpc = kWarps / ks;                       // 8-row groups per CTA pass
  const int g = warp / ks, z = warp - g * ks;
  const int n_groups = (rows + 7) >> 3;
  const int stride = gridDim.x * gpc;
  const int first = blockIdx.x * gpc;
  const int n_pass = first < n_groups ? (n_groups - first + stride - 1) / stride : 0;
  const int per_group = z < nb ? (nb - z + ks - 1) / ks : 0;   // superblocks of this warp per group
  const int n_items = n_pass * per_group;
  uint8_t* ring_base = smem + L.stages + (size_t)warp * ring * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars) + warp * ring;

  if (lane == 0) {
    for (int i = 0; i < ring; ++i) tc::mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // item j of this warp -> group and superblock
  auto item_group = [&](int j) { return first + (j / per_group) * stride + g; };
  auto item_sb = [&](int j) { return z + (j % per_group) * ks; };
  auto issue = [&](int j) {
    const int grp = item_group(j), sb = item_sb(j);
    const int slot = j % ring;
    int n_rows = 0;
    if (grp < n_groups) n_rows = min(8, rows - grp * 8);
    if (lane == 0) tc::mbar_arrive_expect_tx(&bars[slot], (uint32_t)(n_rows * kBlockBytes));
    __syncwarp();
    if (lane < n_rows) {
      const size_t row = (size_t)grp * 8 + lane;
      tc::bulk_g2s(ring_base + slot * kStageBytes + lane * kBlockBytes,
                   w + (row * nb + sb) * kBlockBytes, kBlockBytes, &bars[slot]);
    }
  };

  const int prime = n_items < ring ? n_items : ring;
  for (int j = 0; j < prime; ++j) issue(j);

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Stage the activations: pre-scaled by 2^-p and paired (lo, hi) per chunk.
  for (int i = tid; i < B * cols; i += kThreads) {
    const int b = i / cols, k = i - b * cols;
    const int s = k >> 8, r = k & 255, cc = r >> 6, t = r & 63;
    const int hi = t >> 5, l = t & 31;
    const float scale = __uint_as_float((uint32_t)(127 - nib_shift(l, hi)) << 23);
    xs[(((size_t)b * nb + s) * 4 + cc) * kRegion + 2 * l + hi] = x[(size_t)b * cols + k] * scale;
  }
  // Sums of x over each 32-wide sub-block (fixed order: 8 lanes x 4 values).
  for (int i = warp; i < B * nb * 8 / 4; i += kWarps) {
    const int base = 4 * i;            // four sub-blocks per warp pass, 8 lanes each
    const int sbk = base + (lane >> 3);
    const int b = sbk / (nb * 8), j = sbk - b * nb * 8;
    const float4 v = *reinterpret_cast<const float4*>(x + (size_t)b * cols + 32 * j + 4 * (lane & 7));
    float sum = (v.x + v.y) + (v.z + v.w);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if ((lane & 7) == 0) xsum[sbk] = sum;
  }
  __syncthreads();

  // lane-constant masks for the scale/min decode of sub-blocks 2c, 2c+1
  const int sh = (c & 1) * 16;
  const uint32_t mA = c < 2 ? 0x3F3Fu : 0u, mB = c < 2 ? 0u : 0x0F0Fu, mC = c < 2 ? 0u : 0x3030u;
  const float2 kMagic2 = make_float2(-8388608.0f, -8388608.0f);
  int zero = 0;
  bool ok = true;

  int j = 0;
  for (int pass = 0; pass < n_pass; ++pass) {
    const int grp = first + pass * stride + g;
    const int row = grp * 8 + r8;
    const bool valid = grp < n_groups && row < rows;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    for (int t = 0; t < per_group; ++t, ++j) {
      const int slot = j % ring;
      const int sb = item_sb(j);
      if (ok && !tc::mbar_wait(&bars[slot], (uint32_t)((j / ring) & 1), &zero)) {
        ok = false;
        if (lane == 0) atomicOr(err, 2);
      }
      const uint8_t* st = ring_base + slot * kStageBytes + r8 * kBlockBytes;
      const uint4 hd = *reinterpret_cast<const uint4*>(st);
      const uint4 q0 = *reinterpret_cast<const uint4*>(st + 16 + 32 * c);
      const uint4 q1 = *reinterpret_cast<const uint4*>(st + 32 + 32 * c);
      const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
      const uint32_t a1 = hd.y >> sh, a2 = hd.z >> sh, a3 = hd.w >> sh;
      const uint32_t sc01 = (a1 & mA) | (a3 & mB) | ((a1 >> 2) & mC);
      const uint32_t m01 = (a2 & mA) | ((a3 >> 4) & mB) | ((a2 >> 2) & mC);
      const float sc_lo = (float)(sc01 & 0xFFu), sc_hi = (float)(sc01 >> 8);
      const float m_lo = (float)(m01 & 0xFFu), m_hi = (float)(m01 >> 8);

      float2 pe[B], po[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        pe[b] = make_float2(0.0f, 0.0f);
        po[b] = make_float2(0.0f, 0.0f);
      }
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
                xs + (((size_t)b * nb + sb) * 4 + c) * kRegion + 2 * (16 * h + 4 * k));
            const float4 xa = xp[0], xb = xp[1];
            pe[b] = __ffma2_rn(f0, make_float2(xa.x, xa.y), pe[b]);
            po[b] = __ffma2_rn(f1, make_float2(xa.z, xa.w), po[b]);
            pe[b] = __ffma2_rn(f2, make_float2(xb.x, xb.y), pe[b]);
            po[b] = __ffma2_rn(f3, make_float2(xb.z, xb.w), po[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float2 part = __fadd2_rn(pe[b], po[b]);
        const float2 xsm = *reinterpret_cast<const float2*>(xsum + (size_t)b * nb * 8 + sb * 8 + 2 * c);
        const float scaled = fmaf(sc_hi, part.y, sc_lo * part.x);
        const float mins = fmaf(m_hi, xsm.y, m_lo * xsm.x);
        acc[b] = fmaf(dm.x, scaled, acc[b]);
        acc[b] = fmaf(-dm.y, mins, acc[b]);
      }
      // every lane has used its words of this stage: hand it back to the copy engine
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (j + ring < n_items) issue(j + ring);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
    }
    if (ks == 1) {
      if (valid && c == 0 && ok) {
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
      if (z == 0 && c == 0 && valid && ok) {
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

int pick_ring(int batch, int nb, int smem_optin) {
  for (int ring = 4; ring >= 2; --ring)
    if (layout(batch, nb, ring).total <= (size_t)smem_optin) return ring;
  return 0;
}

template <int B>
cudaError_t launch_b(const uint8_t* w, int rows, int nb, const float* x,
                     const float* residual, float* y, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo& info = device_info(dev);
  const int ring = pick_ring(B, nb, info.max_smem_optin);
  if (ring == 0) return cudaErrorNotSupported;
  const size_t smem = layout(B, nb, ring).total;
  // raise the kernel's dynamic shared-memory limit once per device
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if (limit < info.max_smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_block144_kernel<B>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin);
    if (e != cudaSuccess) return e;
    limit = info.max_smem_optin;
  }
  int* err = device_error_word();
  if (!err) return cudaErrorInvalidValue;
  const int n_groups = (rows + 7) / 8;
  // split K across warps until every SM has a full CTA of work
  int ks = 1;
  while (ks < kWarps && ks * 2 <= nb && (int64_t)n_groups * ks < (int64_t)info.sm_count * kWarps) ks *= 2;
  const int gpc = kWarps / ks;
  int grid = (n_groups + gpc - 1) / gpc;
  if (grid > info.sm_count) grid = info.sm_count;
  gemv_block144_kernel<B><<<grid, kThreads, smem, s>>>(w, rows, nb, ks, ring, x, residual, y, err);
  return cudaGetLastError();
}

}  // namespace

bool gemv_supported(int64_t cols, int batch) {
  if (batch < 1 || batch > 8) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return pick_ring(batch, (int)(cols / kQK), device_info(dev).max_smem_optin) != 0;
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
