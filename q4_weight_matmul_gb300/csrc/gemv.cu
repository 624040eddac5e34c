// q4k_gemv / q4k_gemv_multi: decode GEMV y[b][o] = sum_k w[o][k] x[b][k]
// (+ residual) over BLOCK144 Q4_K weights (genie-ai-runtime §4, Path C: packed
// quants read as whole words, dequantised in registers, residual folded in,
// and one kernel for matrices that share their input: the QKV triple and the
// gate/up pair).
//
// Work split.  Rows are cut into blocks of RB rows (RB = 32, 16 or 8, chosen
// so that the busiest SM holds the fewest rows); one CTA per SM owns a run of
// row blocks (of one or several matrices) and all their superblocks.  A unit
// of work is one row block x one superblock; the 16 consumer warps take units
// round-robin, so K is split across warps.  Each unit leaves one partial sum
// per row in shared memory and the CTA adds a row's partials in superblock
// order (bitwise deterministic).
//
// Streaming.  A producer warp fetches the weights with 3-D tensor copies:
// one copy per stage of RB rows x (128/RB) superblocks (18 KB, out-of-range
// rows and superblocks zero-filled) into a ring of stages.  The copies start
// at launch, before the activations are read.  A CTA stays under half of an
// SM (<= 56 registers per thread, <= ~110 KB of shared memory) so that, when
// launched as a programmatic dependent (opt-in, see pdl_mode), the next
// GEMV's CTA can sit beside it; griddepcontrol.wait orders every activation
// read after the previous kernel has completed.
//
// Lanes.  32/RB lanes share a row: with RB = 32 a lane owns a row's whole
// superblock (256 weights), with RB = 16 half of it, with RB = 8 one 64-weight
// chunk.  A chunk's 32 quant bytes hold sub-block 2c in low nibbles and 2c+1
// in high nibbles.
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
#include <cstdlib>
#include <cstring>

namespace q4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;     // + one producer warp
constexpr int kRegion = 68;                   // floats per (token, superblock, chunk): 32 (lo,hi) pairs + pad
constexpr int kStageSuper = 128;              // superblock-rows per stage (RB * SB)
constexpr int kStageBytes = kStageSuper * kBlockBytes;
constexpr int kMaxRing = 6;
constexpr size_t kPairSmem = 110 * 1024;      // a CTA this small leaves room for a neighbour
constexpr int kMaxMats = 4;

struct GemvParams {
  CUtensorMap map[kMaxMats];
  float* y[kMaxMats];
  const float* res[kMaxMats];
  int rows[kMaxMats];
  int rb_start[kMaxMats + 1];   // prefix sums of row blocks per matrix
  int n_mats;
  int nb, rb_per_cta, rb_pass, ring;
  int trigger_late;             // launch dependents after the units, not at start
  const float* x;
  int* err;
};

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

// which matrix a global row block belongs to
__device__ __forceinline__ int mat_of(const GemvParams& P, int g) {
  int m = 0;
#pragma unroll
  for (int i = 1; i < kMaxMats; ++i)
    if (i < P.n_mats && g >= P.rb_start[i]) m = i;
  return m;
}

// Activations staged once: pre-scaled by 2^-p, (lo, hi)-paired per chunk, and
// summed over each 32-wide sub-block.  All loads of a round are issued before
// any use; eight lanes hold one sub-block, so its sum is three shuffles.
template <int B>
__device__ __forceinline__ void stage_x(const float* __restrict__ x, int nb, float* xs, float* xsum,
                                        int tid) {
  const int row4 = nb * 64;                     // float4 per activation row
  const int n4 = B * row4;                      // a multiple of 64: whole warps
  const float4* x4 = reinterpret_cast<const float4*>(x);
  for (int base = tid; base < n4; base += 4 * kConsumers) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kConsumers;
      if (idx < n4) v[u] = __ldg(x4 + idx);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kConsumers;
      if (idx < n4) {
        const int b = idx / row4, k = 4 * (idx - b * row4);
        const int s = k >> 8, r = k & 255, c = r >> 6, t = r & 63;
        const int hi = t >> 5, l = t & 31;
        float* dst = xs + (((size_t)b * nb + s) * 4 + c) * kRegion + 2 * l + hi;
        // scale exponents of l%4 = 0..3: low half 0, 8, 16, 12; high half 4, 12, 8, 16
        if (hi) {
          dst[0] = v[u].x * 0x1p-4f;
          dst[2] = v[u].y * 0x1p-12f;
          dst[4] = v[u].z * 0x1p-8f;
          dst[6] = v[u].w * 0x1p-16f;
        } else {
          dst[0] = v[u].x;
          dst[2] = v[u].y * 0x1p-8f;
          dst[4] = v[u].z * 0x1p-16f;
          dst[6] = v[u].w * 0x1p-12f;
        }
        float sum = (v[u].x + v[u].y) + (v[u].z + v[u].w);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if ((idx & 7) == 0) xsum[(size_t)b * nb * 8 + (k >> 5)] = sum;
      }
    }
  }
}

// LPR: lanes per row (1, 2 or 4); RB = 32 / LPR rows per block.
template <int B, int LPR>
__global__ void __launch_bounds__(kThreads, (B <= 2 ? 2 : 1)) gemv_block144_kernel(
    const __grid_constant__ GemvParams P) {
  constexpr int RB = 32 / LPR;              // rows per block
  constexpr int SB = kStageSuper / RB;      // superblocks per stage
  constexpr int CPL = 4 / LPR;              // 64-weight chunks per lane
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps every access below in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int nb = P.nb, ring = P.ring, rb_pass = P.rb_pass;
  const int n_rb = P.rb_start[P.n_mats];
  const int rb0 = blockIdx.x * P.rb_per_cta;
  const int my_rb = max(0, min(P.rb_per_cta, n_rb - rb0));
  const int n_sj = (nb + SB - 1) / SB;      // stages per row block
  const int n_stages = my_rb * n_sj;
  const Layout L = layout(B, nb, ring, B * rb_pass * nb * RB);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  float* part = reinterpret_cast<float*>(smem + L.part);      // [B][rb of the pass][nb][RB]
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ring;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // the next kernel in the stream may start its own weight stream now
  if (!P.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
      int slot = 0, g = rb0, sj = 0;
      int m = mat_of(P, g);
      uint32_t phase = 0;
      int issued = 0;
      for (int j = 0; j < n_stages; ++j) {
        if (!tc::mbar_wait_sleep(&empty[slot], phase ^ 1)) {
          atomicOr(P.err, 2);
          break;
        }
        ++issued;
        tc::mbar_arrive_expect_tx(&full[slot], kStageBytes);
        tc::tma_load_3d(stages + (size_t)slot * kStageBytes, &P.map[m], 0, (g - P.rb_start[m]) * RB, sj * SB,
                        &full[slot]);
        if (++sj == n_sj) {
          sj = 0;
          ++g;
          m = mat_of(P, g);
        }
        if (++slot == ring) {
          slot = 0;
          phase ^= 1;
        }
      }
      // every copy issued has landed before this warp (and so the CTA) exits,
      // even if consumers gave up a wait and left early (bounded as well)
      for (int j = max(0, issued - ring); j < issued; ++j)
        if (!tc::mbar_wait_sleep(&full[j % ring], (uint32_t)((j / ring) & 1))) atomicOr(P.err, 2);
    }
    if (P.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x<B>(P.x, nb, xs, xsum, tid);
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
        if (lane == 0) atomicOr(P.err, 2);
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
      const int g = rb0 + pb + rbl;
      const int m = mat_of(P, g);
      const int rows = P.rows[m];
      const int row = (g - P.rb_start[m]) * RB + r;
      if (row < rows && ok) {
        const float* pp = part + (((size_t)b * rb_pass + rbl) * nb) * RB + r;
        float v = 0.0f;
        for (int s2 = 0; s2 < nb; ++s2) v += pp[(size_t)s2 * RB];
        if (P.res[m]) v += P.res[m][(size_t)b * rows + row];
        P.y[m][(size_t)b * rows + row] = v;
      }
    }
    named_sync_consumers();
  }
  if (P.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Programmatic dependent launch (opt-in): Q4K_PDL=1 lets the next kernel
// launch as soon as this one starts, Q4K_PDL=2 once a CTA has finished its
// work, unset or 0 launches normally.  Measured on GB300 for the Qwen3-4B
// decode layer, both PDL modes were slower (59 us vs 42 us per layer), so it
// is off by default.
int pdl_mode() {
  static const int mode = [] {
    const char* v = std::getenv("Q4K_PDL");
    return (v && v[0] >= '0' && v[0] <= '2') ? v[0] - '0' : 0;
  }();
  return mode;
}

struct Plan {
  int lpr, rb_per_cta, rb_pass, grid, ring;
  size_t smem;
};

Plan make_plan(int B, const int64_t* rows, int n_mats, int nb, const DeviceInfo& info) {
  Plan p{};
  // rows per block: the one whose busiest SM holds the fewest rows (ties go to
  // the taller block, which decodes scales less often)
  p.lpr = 4;
  int64_t best = INT64_MAX;
  for (int lpr = 1; lpr <= 4; lpr *= 2) {
    const int64_t rb = 32 / lpr;
    int64_t n_rb = 0;
    for (int m = 0; m < n_mats; ++m) n_rb += (rows[m] + rb - 1) / rb;
    const int64_t per = (n_rb + info.sm_count - 1) / info.sm_count;
    if (per * rb < best) {
      best = per * rb;
      p.lpr = lpr;
    }
  }
  const int RB = 32 / p.lpr;
  int64_t n_rb = 0;
  for (int m = 0; m < n_mats; ++m) n_rb += (rows[m] + RB - 1) / RB;
  p.rb_per_cta = (int)((n_rb + info.sm_count - 1) / info.sm_count);
  p.grid = (int)((n_rb + p.rb_per_cta - 1) / p.rb_per_cta);
  // partial sums of at most 8 KB per pass
  p.rb_pass = (int)std::max<int64_t>(1, std::min<int64_t>(p.rb_per_cta, 2048 / ((int64_t)B * nb * RB)));
  // the deepest ring that keeps the CTA small enough to pair with the next
  // kernel's; failing that, the deepest ring that fits at all
  p.ring = 0;
  const size_t caps[2] = {kPairSmem, (size_t)info.max_smem_optin};
  for (size_t cap : caps) {
    for (int ring = kMaxRing; ring >= 2 && p.ring == 0; --ring) {
      const size_t total = layout(B, nb, ring, B * p.rb_pass * nb * RB).total;
      if (total <= cap) {
        p.ring = ring;
        p.smem = total;
      }
    }
    if (p.ring) break;
  }
  return p;
}

template <int B, int LPR>
cudaError_t launch_bl(const GemvParams& params, const Plan& p, int dev, const DeviceInfo& info,
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_mode() != 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_block144_kernel<B, LPR>, params);
}

template <int B>
cudaError_t launch_b(const uint8_t* const* w, const int64_t* rows, int n_mats, int nb, const float* x,
                     const float* const* residual, float* const* y, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo& info = device_info(dev);
  const Plan p = make_plan(B, rows, n_mats, nb, info);
  if (p.ring == 0) return cudaErrorNotSupported;
  GemvParams params;
  memset(&params, 0, sizeof(params));
  params.err = device_error_word();
  if (!params.err) return cudaErrorInvalidValue;
  const int RB = 32 / p.lpr, SB = kStageSuper / RB;
  params.n_mats = n_mats;
  params.rb_start[0] = 0;
  for (int m = 0; m < n_mats; ++m) {
    // box: a superblock's bytes x RB rows x SB superblocks, rows inner in shared memory
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)rows[m], (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)nb * kBlockBytes, (uint64_t)kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, (uint32_t)RB, (uint32_t)SB};
    if (!encode_tmap_u8_3d(&params.map[m], w[m], dims, strides, box)) return cudaErrorInvalidValue;
    params.y[m] = y[m];
    params.res[m] = residual ? residual[m] : nullptr;
    params.rows[m] = (int)rows[m];
    params.rb_start[m + 1] = params.rb_start[m] + (int)((rows[m] + RB - 1) / RB);
  }
  for (int m = n_mats; m < kMaxMats; ++m) params.rb_start[m + 1] = params.rb_start[m];
  params.nb = nb;
  params.rb_per_cta = p.rb_per_cta;
  params.rb_pass = p.rb_pass;
  params.ring = p.ring;
  params.trigger_late = pdl_mode() == 2 ? 1 : 0;
  params.x = x;
  switch (p.lpr) {
    case 1: return launch_bl<B, 1>(params, p, dev, info, s);
    case 2: return launch_bl<B, 2>(params, p, dev, info, s);
    default: return launch_bl<B, 4>(params, p, dev, info, s);
  }
}

}  // namespace

int gemv_max_mats() { return kMaxMats; }

bool gemv_supported(const int64_t* rows, int n_mats, int64_t cols, int batch) {
  if (batch < 1 || batch > 8 || n_mats < 1 || n_mats > kMaxMats) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  return make_plan(batch, rows, n_mats, (int)(cols / kQK), device_info(dev)).ring != 0;
}

cudaError_t launch_gemv_block144(const uint8_t* const* w, const int64_t* rows, int n_mats, int64_t cols,
                                 const float* x, int batch, const float* const* residual,
                                 float* const* y, cudaStream_t s) {
  const int nb = (int)(cols / kQK);
  switch (batch) {
    case 1: return launch_b<1>(w, rows, n_mats, nb, x, residual, y, s);
    case 2: return launch_b<2>(w, rows, n_mats, nb, x, residual, y, s);
    case 3: return launch_b<3>(w, rows, n_mats, nb, x, residual, y, s);
    case 4: return launch_b<4>(w, rows, n_mats, nb, x, residual, y, s);
    case 5: return launch_b<5>(w, rows, n_mats, nb, x, residual, y, s);
    case 6: return launch_b<6>(w, rows, n_mats, nb, x, residual, y, s);
    case 7: return launch_b<7>(w, rows, n_mats, nb, x, residual, y, s);
    case 8: return launch_b<8>(w, rows, n_mats, nb, x, residual, y, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace q4k
