// q4k_gemv: decode GEMV y[b][o] = sum_k w[o][k] x[b][k] (+ residual) over
// BLOCK144 Q4_K weights (genie-ai-runtime §4, Path C: packed quants read as
// whole words, dequantised in registers, residual folded in).
//
// Streaming.  One persistent CTA per SM: a producer warp and 16 consumer
// warps.  The matrix is cut into tiles of `tr` rows; a tile streams through a
// ring of shared-memory stages, each stage one TMA box of tr rows x S
// superblocks (tr * S = 128, 18 KB), fetched by a single 3-D tensor copy with
// out-of-range rows and superblocks zero-filled.  The producer starts the
// stream at launch, before the activations are staged, and keeps every free
// stage filled; bytes in flight are set by the ring, not by registers.
//
// Mapping.  Consumer warp (g, z) owns 8-row group g of the tile and superblock
// z of each stage; lane (r, c) = (lane/4, lane%4) works on row r and the
// 64-weight chunk c of that superblock (its 32 quant bytes hold all of
// sub-block 2c in low nibbles and 2c+1 in high nibbles).  The S partial sums of
// a group are added in shared memory in a fixed order, so results are
// bitwise deterministic.
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
#include "tmap.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;     // + one producer warp
constexpr int kRegion = 68;                   // floats per (token, superblock, chunk): 32 (lo,hi) pairs + pad
constexpr int kStageSuper = 128;              // superblock-rows per stage (tr * S)
constexpr int kStageBytes = kStageSuper * kBlockBytes;

__device__ __forceinline__ float magic(uint32_t bits) { return __uint_as_float(0x4B000000u | bits); }

// Power-of-two pre-scale exponent of weight l (0..31) of the low (hi = 0) or
// high (hi = 1) half of a chunk; matches the nibble positions used below.
__device__ __forceinline__ int nib_shift(int l, int hi) {
  const uint32_t lo_tab = 0u | (8u << 8) | (16u << 16) | (12u << 24);
  const uint32_t hi_tab = 4u | (12u << 8) | (8u << 16) | (16u << 24);
  return (int)(((hi ? hi_tab : lo_tab) >> (8 * (l & 3))) & 0xFFu);
}

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

struct Layout {
  size_t xs, xsum, red, stages, bars, total;
};

__host__ __device__ inline Layout layout(int B, int nb, int ring) {
  Layout L;
  L.xs = 0;
  L.xsum = L.xs + sizeof(float) * (size_t)B * nb * 4 * kRegion;
  L.red = L.xsum + sizeof(float) * (size_t)B * nb * 8;
  L.stages = (L.red + sizeof(float) * (size_t)kConsumerWarps * 8 * B + 1023) & ~size_t(1023);
  L.bars = L.stages + (size_t)ring * kStageBytes;
  L.total = L.bars + sizeof(uint64_t) * 2 * ring + 1024;   // + slack to align the base
  return L;
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_block144_kernel(
    const __grid_constant__ CUtensorMap tmap, int rows, int nb, int tr, int ring, int rows_inner,
    const float* __restrict__ x, const float* __restrict__ residual,
    float* __restrict__ y, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout L = layout(B, nb, ring);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ring;

  const int cols = nb * kQK;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = kStageSuper / tr;                    // superblocks per stage
  const int n_tiles = (rows + tr - 1) / tr;
  const int n_st = (nb + S - 1) / S;                 // stages per tile

  if (tid == 0) {
    for (int i = 0; i < ring; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap) : "memory");
      int slot = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        for (int st = 0; st < n_st; ++st) {
          if (!tc::mbar_wait_sleep(&empty[slot], phase ^ 1)) {
            atomicOr(err, 2);
            return;
          }
          tc::mbar_arrive_expect_tx(&full[slot], kStageBytes);
          if (rows_inner)
            tc::tma_load_3d(stages + (size_t)slot * kStageBytes, &tmap, 0, tile * tr, st * S, &full[slot]);
          else
            tc::tma_load_3d(stages + (size_t)slot * kStageBytes, &tmap, 0, st * S, tile * tr, &full[slot]);
          if (++slot == ring) {
            slot = 0;
            phase ^= 1;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Stage the activations: pre-scaled by 2^-p and paired (lo, hi) per chunk.
  for (int i = tid; i < B * cols; i += kConsumers) {
    const int b = i / cols, k = i - b * cols;
    const int s = k >> 8, r = k & 255, cc = r >> 6, t = r & 63;
    const int hi = t >> 5, l = t & 31;
    const float scale = __uint_as_float((uint32_t)(127 - nib_shift(l, hi)) << 23);
    xs[(((size_t)b * nb + s) * 4 + cc) * kRegion + 2 * l + hi] = x[(size_t)b * cols + k] * scale;
  }
  // Sums of x over each 32-wide sub-block (fixed order: 8 lanes x 4 values).
  for (int i = warp; i < B * nb * 2; i += kConsumerWarps) {
    const int sbk = 4 * i + (lane >> 3);
    const int b = sbk / (nb * 8), j = sbk - b * nb * 8;
    const float4 v = *reinterpret_cast<const float4*>(x + (size_t)b * cols + 32 * j + 4 * (lane & 7));
    float sum = (v.x + v.y) + (v.z + v.w);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if ((lane & 7) == 0) xsum[sbk] = sum;
  }
  named_sync_consumers();

  const int g = warp / S, z = warp - g * S;
  const int r8 = lane >> 2, c = lane & 3;
  const int sh = (c & 1) * 16;
  const uint32_t mA = c < 2 ? 0x3F3Fu : 0u, mB = c < 2 ? 0u : 0x0F0Fu, mC = c < 2 ? 0u : 0x3030u;
  const float2 kMagic2 = make_float2(-8388608.0f, -8388608.0f);
  // this lane's 144-byte superblock inside a stage laid out [S][tr][144]
  // (rows inner) or [tr][S][144]
  const size_t lane_off = rows_inner ? ((size_t)z * tr + g * 8 + r8) * kBlockBytes
                                     : ((size_t)(g * 8 + r8) * S + z) * kBlockBytes;
  bool ok = true;
  int slot = 0;
  uint32_t phase = 0;

  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int row = tile * tr + g * 8 + r8;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    for (int st = 0; st < n_st; ++st) {
      const int sb = st * S + z;
      if (ok && !tc::mbar_wait_sleep(&full[slot], phase)) {
        ok = false;
        if (lane == 0) atomicOr(err, 2);
      }
      if (sb < nb) {
        const uint8_t* p = stages + (size_t)slot * kStageBytes + lane_off;
        const uint4 hd = *reinterpret_cast<const uint4*>(p);
        const uint4 q0 = *reinterpret_cast<const uint4*>(p + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(p + 32 + 32 * c);
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
        const float* xb0 = xs + ((size_t)sb * 4 + c) * kRegion;
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
                  xb0 + (size_t)b * nb * 4 * kRegion + 2 * (16 * h + 4 * k));
              const float4 xa = xp[0], xc = xp[1];
              pe[b] = __ffma2_rn(f0, make_float2(xa.x, xa.y), pe[b]);
              po[b] = __ffma2_rn(f1, make_float2(xa.z, xa.w), po[b]);
              pe[b] = __ffma2_rn(f2, make_float2(xc.x, xc.y), pe[b]);
              po[b] = __ffma2_rn(f3, make_float2(xc.z, xc.w), po[b]);
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
      }
      // release the stage once every lane of the warp has read it
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      if (++slot == ring) {
        slot = 0;
        phase ^= 1;
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
    }
    const bool valid = row < rows && ok;
    if (S == 1) {
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
      named_sync_consumers();
      if (z == 0 && c == 0 && valid) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
          float v = 0.0f;
          for (int zz = 0; zz < S; ++zz) v += red[((warp + zz) * 8 + r8) * B + b];
          if (residual) v += residual[(size_t)b * rows + row];
          y[(size_t)b * rows + row] = v;
        }
      }
      named_sync_consumers();
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

int pick_ring(int batch, int nb, int smem_optin) {
  for (int ring = 4; ring >= 2; --ring)
    if (layout(batch, nb, ring).total <= (size_t)smem_optin) return ring;
  return 0;
}

int pick_tile_rows(int64_t rows, int sm_count) {
  for (int tr = kStageSuper; tr > 8; tr >>= 1)
    if ((rows + tr - 1) / tr >= sm_count) return tr;
  return 8;
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
  const int tr = pick_tile_rows(rows, info.sm_count);
  const int S = kStageSuper / tr;
  // Preferred box order: bytes, rows, superblocks (rows inner: conflict-free
  // shared-memory reads); fall back to the memory order if the driver
  // rejects the non-monotonic strides.
  CUtensorMap map;
  int rows_inner = 1;
  {
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)nb * kBlockBytes, (uint64_t)kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, (uint32_t)tr, (uint32_t)S};
    if (!encode_tmap_u8_3d(&map, w, dims, strides, box)) {
      rows_inner = 0;
      const uint64_t dims2[3] = {(uint64_t)kBlockBytes, (uint64_t)nb, (uint64_t)rows};
      const uint64_t strides2[2] = {(uint64_t)kBlockBytes, (uint64_t)nb * kBlockBytes};
      const uint32_t box2[3] = {(uint32_t)kBlockBytes, (uint32_t)S, (uint32_t)tr};
      if (!encode_tmap_u8_3d(&map, w, dims2, strides2, box2)) return cudaErrorInvalidValue;
    }
  }
  const int n_tiles = (rows + tr - 1) / tr;
  const int grid = n_tiles < info.sm_count ? n_tiles : info.sm_count;
  gemv_block144_kernel<B><<<grid, kThreads, smem, s>>>(map, rows, nb, tr, ring, rows_inner, x, residual,
                                                       y, err);
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
