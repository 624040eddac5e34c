// q4k_gemv: decode GEMV y[b][o] = sum_k w[o][k] x[b][k] (+ residual) over
// BLOCK144 Q4_K weights (genie-ai-runtime §4, Path C: packed quants read as
// whole words, dequantised in registers, residual folded in).
//
// Work split.  Rows are cut into blocks of RB rows (RB = 32, 16 or 8, the
// largest that still gives every SM a block); one CTA per SM owns a run of
// row blocks and all their superblocks.  A unit of work is one row block x
// one superblock; the 16 consumer warps of a CTA take units round-robin, so
// every warp streams several superblocks and K is split across warps.  Each
// unit leaves one partial sum per row in shared memory; at the end the CTA
// adds a row's partials in superblock order (bitwise deterministic).
//
// Streaming.  A producer warp fetches the CTA's weights with 3-D tensor
// copies: one copy per stage of RB rows x (128/RB) superblocks (18 KB, out of
// range rows and superblocks zero-filled) into a ring of stages.  It starts
// at launch, before the activations are staged, so bytes in flight are set by
// the ring, not by registers.
//
// Lanes.  32/RB lanes share a row: with RB = 32 a lane owns a row's whole
// superblock (256 weights), with RB = 16 half of it, with RB = 8 one 64-weight
// chunk.  A chunk's 32 quant bytes hold sub-block 2c in low nibbles and 2c+1
// in high nibbles, so scale/min decoding is paid once per 64-256 weights.
//
// Dequantisation.  A nibble at bit position p (p <= 16) ORed into the float
// 2^23 gives 2^23 + q*2^p exactly; subtracting 2^23 leaves q*2^p, and the
// activation staged for that position is pre-multiplied by 2^-p, so the
// product is exactly q*x before its fp32 rounding.  A word of eight nibbles
// costs one shift, eight LOP3s, four fp32x2 adds and four fp32x2 FMAs (per
// token), written in PTX so that the pairs are formed in place.  Per
// sub-block j:  acc += d*sc_j*P_j - dmin*m_j*X_j  with X_j = sum of x over j.
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

namespace q4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;     // + one producer warp
constexpr int kRegion = 68;                   // floats per (token, superblock, chunk): 32 (lo,hi) pairs + pad
constexpr int kStageSuper = 128;              // superblock-rows per stage (RB * SB)
constexpr int kStageBytes = kStageSuper * kBlockBytes;
constexpr int kMaxRing = 8;

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

// Eight nibbles of v -> four exact (q_lo*2^p, q_hi*2^p) fp32 pairs.
__device__ __forceinline__ void conv_word(uint32_t v, uint64_t& f0, uint64_t& f1, uint64_t& f2,
                                          uint64_t& f3) {
  asm("{\n\t.reg .b32 a0,a1,a2,a3,a4,a5,a6,a7,v12;\n\t"
      "shr.b32 v12, %4, 12;\n\t"
      "lop3.b32 a0, %4, 0xF, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a1, %4, 0xF0, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a2, %4, 0xF00, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a3, %4, 0xF000, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a4, %4, 0xF0000, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a5, v12, 0xF00, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a6, v12, 0xF000, 0x4B000000, 0xEA;\n\t"
      "lop3.b32 a7, v12, 0xF0000, 0x4B000000, 0xEA;\n\t"
      "mov.b64 %0, {a0, a1};\n\tmov.b64 %1, {a2, a3};\n\tmov.b64 %2, {a4, a5};\n\tmov.b64 %3, {a6, a7};\n\t"
      "add.rn.f32x2 %0, %0, %5;\n\tadd.rn.f32x2 %1, %1, %5;\n\t"
      "add.rn.f32x2 %2, %2, %5;\n\tadd.rn.f32x2 %3, %3, %5;\n\t}"
      : "=l"(f0), "=l"(f1), "=l"(f2), "=l"(f3)
      : "r"(v), "l"(0xCB000000CB000000ull));
}

// pe += f0*x(0,1) + f2*x(4,5); po += f1*x(2,3) + f3*x(6,7)
__device__ __forceinline__ void fma_word(uint64_t f0, uint64_t f1, uint64_t f2, uint64_t f3,
                                         const uint4& xa, const uint4& xc, uint64_t& pe, uint64_t& po) {
  asm("{\n\t.reg .b64 x0,x1,x2,x3;\n\t"
      "mov.b64 x0, {%6, %7};\n\tmov.b64 x1, {%8, %9};\n\t"
      "mov.b64 x2, {%10, %11};\n\tmov.b64 x3, {%12, %13};\n\t"
      "fma.rn.f32x2 %0, %2, x0, %0;\n\tfma.rn.f32x2 %1, %3, x1, %1;\n\t"
      "fma.rn.f32x2 %0, %4, x2, %0;\n\tfma.rn.f32x2 %1, %5, x3, %1;\n\t}"
      : "+l"(pe), "+l"(po)
      : "l"(f0), "l"(f1), "l"(f2), "l"(f3), "r"(xa.x), "r"(xa.y), "r"(xa.z), "r"(xa.w), "r"(xc.x),
        "r"(xc.y), "r"(xc.z), "r"(xc.w));
}

__device__ __forceinline__ float2 u64_as_f2(uint64_t v) {
  return make_float2(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
}

// byte i of w as a float (exact)
__device__ __forceinline__ float byte_f(uint32_t w, int i) { return (float)((w >> (8 * i)) & 0xFFu); }

struct Layout {
  size_t xs, xsum, part, stages, bars, total;
};

__host__ __device__ inline Layout layout(int B, int nb, int ring, int part_floats) {
  Layout L;
  L.xs = 0;
  L.xsum = L.xs + sizeof(float) * (size_t)B * nb * 4 * kRegion;
  L.part = L.xsum + sizeof(float) * (size_t)B * nb * 8;
  L.stages = (L.part + sizeof(float) * (size_t)part_floats + 1023) & ~size_t(1023);
  L.bars = L.stages + (size_t)ring * kStageBytes;
  L.total = L.bars + sizeof(uint64_t) * 2 * ring + 1024;   // + slack to align the base
  return L;
}

// LPR: lanes per row (1, 2 or 4); RB = 32 / LPR rows per block.
template <int B, int LPR>
__global__ void __launch_bounds__(kThreads, 1) gemv_block144_kernel(
    const __grid_constant__ CUtensorMap tmap, int rows, int nb, int rb_per_cta, int rb_pass, int ring,
    const float* __restrict__ x, const float* __restrict__ residual,
    float* __restrict__ y, int* __restrict__ err) {
  constexpr int RB = 32 / LPR;              // rows per block
  constexpr int SB = kStageSuper / RB;      // superblocks per stage
  constexpr int CPL = 4 / LPR;              // 64-weight chunks per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_rb = (rows + RB - 1) / RB;
  const int rb0 = blockIdx.x * rb_per_cta;
  const int my_rb = max(0, min(rb_per_cta, n_rb - rb0));
  const int n_sj = (nb + SB - 1) / SB;      // stages per row block
  const int n_stages = my_rb * n_sj;
  const Layout L = layout(B, nb, ring, B * rb_pass * nb * RB);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  float* part = reinterpret_cast<float*>(smem + L.part);      // [B][rb of the pass][nb][RB]
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ring;

  const int cols = nb * kQK;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < ring; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], SB);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap) : "memory");
      int slot = 0, rb = 0, sj = 0;
      uint32_t phase = 0;
      for (int j = 0; j < n_stages; ++j) {
        if (!tc::mbar_wait_sleep(&empty[slot], phase ^ 1)) {
          atomicOr(err, 2);
          break;
        }
        tc::mbar_arrive_expect_tx(&full[slot], kStageBytes);
        tc::tma_load_3d(stages + (size_t)slot * kStageBytes, &tmap, 0, (rb0 + rb) * RB, sj * SB, &full[slot]);
        if (++sj == n_sj) {
          sj = 0;
          ++rb;
        }
        if (++slot == ring) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = tid; i < B * cols; i += kConsumers) {
    const int b = i / cols, k = i - b * cols;
    const int s = k >> 8, r = k & 255, cc = r >> 6, t = r & 63;
    const int hi = t >> 5, l = t & 31;
    const float scale = __uint_as_float((uint32_t)(127 - nib_shift(l, hi)) << 23);
    xs[(((size_t)b * nb + s) * 4 + cc) * kRegion + 2 * l + hi] = x[(size_t)b * cols + k] * scale;
  }
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

  const int r_in = lane / LPR;              // row inside the block
  const int lq = lane % LPR;                // this lane's share of the superblock
  const int c0 = lq * CPL;                  // first chunk of the lane
  bool ok = true;
  // Row blocks are processed in passes of at most rb_pass blocks (bounded
  // partial-sum buffer).  Within a pass, unit u = warp, warp + 16, ... lies in
  // stage j = j0 + u / SB at superblock slot z = u % SB.
  for (int pb = 0; pb < my_rb; pb += rb_pass) {
    const int n_rbp = min(rb_pass, my_rb - pb);
    const int j0 = pb * n_sj;
    const int n_units = n_rbp * n_sj * SB;
    for (int u = warp; u < n_units; u += kConsumerWarps) {
      const int jl = u / SB, z = u - jl * SB;
      const int j = j0 + jl;
      const int slot = j % ring;
      const uint32_t phase = (uint32_t)((j / ring) & 1);
      const int rbl = jl / n_sj, sj = jl - rbl * n_sj;
      const int sb = sj * SB + z;
      if (ok && !tc::mbar_wait_sleep(&full[slot], phase)) {
        ok = false;
        if (lane == 0) atomicOr(err, 2);
      }
      float acc[B];
#pragma unroll
      for (int b = 0; b < B; ++b) acc[b] = 0.0f;
      if (sb < nb) {
        // stage laid out [SB][RB][144] (rows inner)
        const uint8_t* p = stages + (size_t)slot * kStageBytes + ((size_t)z * RB + r_in) * kBlockBytes;
        const uint4 hd = *reinterpret_cast<const uint4*>(p);
        const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
        // scales (sc) and mins (m) of sub-blocks 0..3 and 4..7, one byte each
        const uint32_t sc03 = hd.y & 0x3F3F3F3Fu, m03 = hd.z & 0x3F3F3F3Fu;
        const uint32_t sc47 = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        const uint32_t m47 = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
        float scaled[B], mins[B];
#pragma unroll
        for (int b = 0; b < B; ++b) scaled[b] = mins[b] = 0.0f;
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) {
          const int c = c0 + cc;
          const uint4 q0 = *reinterpret_cast<const uint4*>(p + 16 + 32 * c);
          const uint4 q1 = *reinterpret_cast<const uint4*>(p + 32 + 32 * c);
          uint64_t pe[B], po[B];
#pragma unroll
          for (int b = 0; b < B; ++b) pe[b] = po[b] = 0ull;
          const float* xc0 = xs + ((size_t)sb * 4 + c) * kRegion;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 qq = h ? q1 : q0;
            const uint32_t words[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint64_t f0, f1, f2, f3;
              conv_word(words[k], f0, f1, f2, f3);
#pragma unroll
              for (int b = 0; b < B; ++b) {
                const uint4* xp =
                    reinterpret_cast<const uint4*>(xc0 + (size_t)b * nb * 4 * kRegion + 2 * (16 * h + 4 * k));
                fma_word(f0, f1, f2, f3, xp[0], xp[1], pe[b], po[b]);
              }
            }
          }
          // sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)
          const uint32_t scw = c < 2 ? sc03 : sc47, mw = c < 2 ? m03 : m47;
          const int bi = 2 * (c & 1);
          const float sc_lo = byte_f(scw, bi), sc_hi = byte_f(scw, bi + 1);
          const float m_lo = byte_f(mw, bi), m_hi = byte_f(mw, bi + 1);
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const float2 a = u64_as_f2(pe[b]), o = u64_as_f2(po[b]);
            const float2 xsm = *reinterpret_cast<const float2*>(xsum + (size_t)b * nb * 8 + sb * 8 + 2 * c);
            scaled[b] = fmaf(sc_hi, a.y + o.y, fmaf(sc_lo, a.x + o.x, scaled[b]));
            mins[b] = fmaf(m_hi, xsm.y, fmaf(m_lo, xsm.x, mins[b]));
          }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = fmaf(dm.x, scaled[b], -dm.y * mins[b]);
      }
      // release the stage once every lane of the warp has read it
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (LPR >= 2) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
        if (LPR >= 4) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
      }
      if (lq == 0 && sb < nb) {
#pragma unroll
        for (int b = 0; b < B; ++b) part[(((size_t)b * rb_pass + rbl) * nb + sb) * RB + r_in] = acc[b];
      }
    }
    named_sync_consumers();
    // y = sum of a row's partials in superblock order (+ residual)
    for (int i = tid; i < B * n_rbp * RB; i += kConsumers) {
      const int b = i / (n_rbp * RB), rem = i - b * n_rbp * RB;
      const int rbl = rem / RB, r = rem - rbl * RB;
      const int row = (rb0 + pb + rbl) * RB + r;
      if (row < rows && ok) {
        const float* pp = part + (((size_t)b * rb_pass + rbl) * nb) * RB + r;
        float v = 0.0f;
        for (int s2 = 0; s2 < nb; ++s2) v += pp[(size_t)s2 * RB];
        if (residual) v += residual[(size_t)b * rows + row];
        y[(size_t)b * rows + row] = v;
      }
    }
    named_sync_consumers();
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct Plan {
  int lpr, rb_per_cta, rb_pass, grid, ring;
  size_t smem;
};

Plan make_plan(int B, int64_t rows, int nb, const DeviceInfo& info) {
  Plan p{};
  // rows per block: the one whose busiest SM holds the fewest rows (ties go to
  // the taller block, which decodes scales less often)
  p.lpr = 4;
  int64_t best = INT64_MAX;
  for (int lpr = 1; lpr <= 4; lpr *= 2) {
    const int64_t rb = 32 / lpr, n_rb = (rows + rb - 1) / rb;
    const int64_t per = (n_rb + info.sm_count - 1) / info.sm_count;
    if (per * rb < best) {
      best = per * rb;
      p.lpr = lpr;
    }
  }
  const int RB = 32 / p.lpr;
  const int n_rb = (int)((rows + RB - 1) / RB);
  p.rb_per_cta = (n_rb + info.sm_count - 1) / info.sm_count;
  p.grid = (n_rb + p.rb_per_cta - 1) / p.rb_per_cta;
  // partial sums of at most 16 KB per pass
  p.rb_pass = (int)std::max<int64_t>(1, std::min<int64_t>(p.rb_per_cta, 4096 / ((int64_t)B * nb * RB)));
  p.ring = 0;
  for (int ring = kMaxRing; ring >= 2; --ring) {
    const size_t total = layout(B, nb, ring, B * p.rb_pass * nb * RB).total;
    if (total <= (size_t)info.max_smem_optin) {
      p.ring = ring;
      p.smem = total;
      break;
    }
  }
  return p;
}

template <int B, int LPR>
cudaError_t launch_bl(const CUtensorMap& map, int rows, int nb, const Plan& p, const float* x,
                      const float* residual, float* y, int* err, int dev, const DeviceInfo& info,
                      cudaStream_t s) {
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if (limit < info.max_smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_block144_kernel<B, LPR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin);
    if (e != cudaSuccess) return e;
    limit = info.max_smem_optin;
  }
  gemv_block144_kernel<B, LPR><<<p.grid, kThreads, p.smem, s>>>(map, rows, nb, p.rb_per_cta, p.rb_pass,
                                                                p.ring, x, residual, y, err);
  return cudaGetLastError();
}

template <int B>
cudaError_t launch_b(const uint8_t* w, int rows, int nb, const float* x,
                     const float* residual, float* y, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo& info = device_info(dev);
  const Plan p = make_plan(B, rows, nb, info);
  if (p.ring == 0) return cudaErrorNotSupported;
  int* err = device_error_word();
  if (!err) return cudaErrorInvalidValue;
  const int RB = 32 / p.lpr, SB = kStageSuper / RB;
  // box: bytes of a superblock x RB rows x SB superblocks, rows inner in shared memory
  CUtensorMap map;
  const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)rows, (uint64_t)nb};
  const uint64_t strides[2] = {(uint64_t)nb * kBlockBytes, (uint64_t)kBlockBytes};
  const uint32_t box[3] = {(uint32_t)kBlockBytes, (uint32_t)RB, (uint32_t)SB};
  if (!encode_tmap_u8_3d(&map, w, dims, strides, box)) return cudaErrorInvalidValue;
  switch (p.lpr) {
    case 1: return launch_bl<B, 1>(map, rows, nb, p, x, residual, y, err, dev, info, s);
    case 2: return launch_bl<B, 2>(map, rows, nb, p, x, residual, y, err, dev, info, s);
    default: return launch_bl<B, 4>(map, rows, nb, p, x, residual, y, err, dev, info, s);
  }
}

}  // namespace

bool gemv_supported(int64_t rows, int64_t cols, int batch) {
  if (batch < 1 || batch > 8) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return make_plan(batch, rows, (int)(cols / kQK), device_info(dev)).ring != 0;
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
