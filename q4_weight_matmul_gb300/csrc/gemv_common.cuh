// Device arithmetic shared by the decode GEMV kernels (gemv.cu, gemv_seq.cu):
// the fixed-point staging of the activations and the dot product of one
// lane's share of a Q4_K superblock with them (genie-ai-runtime §4, Path C:
// quants read as whole words and dequantised in registers).
//
// Activations.  Each 32-wide sub-block j of x is held as a 23-bit fixed-point
// integer X = rint(x / s_j) with a power-of-two scale s_j = 2^(e-22), e the
// exponent of the sub-block's largest |x| (so |X| <= 2^22 and
// |x - s_j*X| <= s_j/2 <= 2^-22 * max|x|), split into three byte planes
// X = 65536*X2 + 256*X1 + X0 (X0, X1 unsigned, X2 signed).  The 4-bit quants
// q enter dp4a dot products with the planes unchanged, so P_j = sum q*X over
// the sub-block is an exact integer; the per-sub-block scales are applied in
// fp32 registers:
//     acc += d*sc_j*s_j*P_j - dmin*m_j*XS_j,    XS_j = sum of x over j.
// A 32-bit word of quants (8 weights) costs a shift, two LOP3s and six dp4a
// per token, against one fp32 multiply-add per weight for a dequantised dot.
#pragma once

#include "q4k_internal.h"
#include "tc_ptx.cuh"

#include <cuda_fp16.h>
#include <cstdint>

namespace q4k {
namespace gemv {

constexpr int kRegion = 208;   // bytes per (token, superblock, chunk) of x planes: 192 + pad

// acc += dot of the four unsigned bytes of a and of b
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int acc) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(acc));
  return d;
}
// acc += dot of the four unsigned bytes of a and the four signed bytes of b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int acc) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(acc));
  return d;
}

// byte i of w as a float (exact)
__device__ __forceinline__ float byte_f(uint32_t w, int i) { return (float)((w >> (8 * i)) & 0xFFu); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// Bounded spin until a producer has issued stage j of its ring (false on
// timeout).  A consumer that skips stages must see stage j issued before it
// waits on the stage's parity: the copy of stage j - ring (same slot, same
// parity two phases back) may still be in flight, and a parity wait would
// then pass on the old phase.
__device__ __noinline__ inline bool wait_issued(volatile int* issued, int j) {
  const long long t0 = clock64();
  while (*issued <= j) {
    __nanosleep(64);
    if (clock64() - t0 > tc::kTimeoutCycles) return false;
  }
  return true;
}

// Shared-memory bytes of the staged activations: planes, then (scale, sum)
// pairs per sub-block.
__host__ __device__ constexpr size_t xs_bytes(int B, int nb) { return (size_t)B * nb * 4 * kRegion; }
__host__ __device__ constexpr size_t xss_bytes(int B, int nb) { return sizeof(float2) * (size_t)B * nb * 8; }

// Stage x [B][nb*256] once per CTA as byte planes of 23-bit fixed point, with
// each sub-block's scale s_j and fp32 sum XS_j.  Eight lanes hold one
// sub-block (four elements each), so its max and sum are three shuffles; all
// loads of a round are issued before any use.  NT threads (a multiple of 32,
// tid < NT) take part.  kCoherent reads x through L2 only (x may have been
// written earlier in the same kernel); otherwise through the read-only path.
// Plane layout per (token, superblock, chunk c): 16-byte words at
// ((h*3 + p)*2 + s)*16, h = half of the chunk's 32 positions, p = plane,
// s = sub-block 2c (0) or 2c+1 (1); word k of it holds positions 16h+4k..+3.
template <int B, int NT, bool kCoherent>
__device__ __forceinline__ void stage_x(const float* __restrict__ x, int nb, uint8_t* xs, float2* xss,
                                        int tid) {
  const int row4 = nb * 64;                     // float4 per activation row
  const int n4 = B * row4;                      // a multiple of 64: whole warps
  const float4* x4 = reinterpret_cast<const float4*>(x);
  for (int base = tid; base < n4; base += 5 * NT) {
    float4 v[5];
#pragma unroll
    for (int u = 0; u < 5; ++u) {
      const int idx = base + u * NT;
      if (idx < n4) v[u] = kCoherent ? __ldcg(x4 + idx) : __ldg(x4 + idx);
    }
#pragma unroll
    for (int u = 0; u < 5; ++u) {
      const int idx = base + u * NT;
      if (idx < n4) {
        const int b = idx / row4, k = 4 * (idx - b * row4);
        const int sb = k >> 8, r = k & 255, j = r >> 5, pos = r & 31;
        const int c = j >> 1, sf = j & 1, h = pos >> 4, kw = (pos & 15) >> 2;
        float amax = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
        float sum = (v[u].x + v[u].y) + (v[u].z + v[u].w);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        // power-of-two scale: |x| < 2^(E-126) for the biased exponent E of
        // amax, so X = rint(x * 2^(148-E)) satisfies |X| <= 2^22; blocks
        // below 2^-104 (and all-zero blocks) are staged as zero
        const int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
        const bool live = E >= 22;
        const float mul = live ? __uint_as_float((uint32_t)(275 - E) << 23) : 0.0f;
        const float scale = live ? __uint_as_float((uint32_t)(E - 21) << 23) : 0.0f;
        const int X0 = __float2int_rn(v[u].x * mul), X1 = __float2int_rn(v[u].y * mul);
        const int X2 = __float2int_rn(v[u].z * mul), X3 = __float2int_rn(v[u].w * mul);
        uint32_t* dst = reinterpret_cast<uint32_t*>(xs + (((size_t)b * nb + sb) * 4 + c) * kRegion) +
                        (h * 3 * 2 + sf) * 4 + kw;
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
          const int sh = 8 * pl;
          const uint32_t word = ((uint32_t)(X0 >> sh) & 0xFFu) | (((uint32_t)(X1 >> sh) & 0xFFu) << 8) |
                                (((uint32_t)(X2 >> sh) & 0xFFu) << 16) | (((uint32_t)(X3 >> sh) & 0xFFu) << 24);
          dst[pl * 2 * 4] = word;
        }
        if ((idx & 7) == 0) xss[((size_t)b * nb + sb) * 8 + j] = make_float2(scale, sum);
      }
    }
  }
}

// One lane's share of one superblock row against the staged activations:
// chunks c0 .. c0+CPL-1 (64 weights each) of the BLOCK144 superblock at `p`
// (shared memory), superblock index sb of x.  acc[b] receives
// d * sum_j sc_j s_j P_j - dmin * sum_j m_j XS_j over the lane's sub-blocks.
template <int B, int CPL>
__device__ __forceinline__ void superblock_dot(const uint8_t* p, const uint8_t* xs, const float2* xss, int nb,
                                               int sb, int c0, float (&acc)[B]) {
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
    // exact integer sums of q * X per plane, low (sub-block 2c) and high
    // (2c+1) nibbles
    int lo[B][3], hi[B][3];
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
      for (int pl = 0; pl < 3; ++pl) lo[b][pl] = hi[b][pl] = 0;
    const uint8_t* xc0 = xs + ((size_t)sb * 4 + c) * kRegion;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 qq = h ? q1 : q0;
      uint32_t ql[4], qh[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = word_of(qq, k);
        ql[k] = w & 0x0F0F0F0Fu;
        qh[k] = (w >> 4) & 0x0F0F0F0Fu;
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint4* xp = reinterpret_cast<const uint4*>(xc0 + (size_t)b * nb * 4 * kRegion) + h * 6;
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
          const uint4 xl = xp[2 * pl], xh = xp[2 * pl + 1];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (pl < 2) {
              lo[b][pl] = dp4a_uu(ql[k], word_of(xl, k), lo[b][pl]);
              hi[b][pl] = dp4a_uu(qh[k], word_of(xh, k), hi[b][pl]);
            } else {
              lo[b][pl] = dp4a_us(ql[k], word_of(xl, k), lo[b][pl]);
              hi[b][pl] = dp4a_us(qh[k], word_of(xh, k), hi[b][pl]);
            }
          }
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
      // P = 65536*P2 + (256*P1 + P0); the bracket is an exact int32
      const float p_lo = fmaf((float)lo[b][2], 65536.0f, (float)(lo[b][1] * 256 + lo[b][0]));
      const float p_hi = fmaf((float)hi[b][2], 65536.0f, (float)(hi[b][1] * 256 + hi[b][0]));
      const float4 ss = *reinterpret_cast<const float4*>(xss + ((size_t)b * nb + sb) * 8 + 2 * c);
      scaled[b] = fmaf(sc_hi * ss.z, p_hi, fmaf(sc_lo * ss.x, p_lo, scaled[b]));
      mins[b] = fmaf(m_hi, ss.w, fmaf(m_lo, ss.y, mins[b]));
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = fmaf(dm.x, scaled[b], -dm.y * mins[b]);
}

}  // namespace gemv
}  // namespace q4k
