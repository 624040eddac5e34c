// Device arithmetic shared by the decode GEMV kernels (gemv.cu, gemv_seq.cu):
// the fixed-point staging of the activations and the dot product of one
// lane's share of a Q4_K superblock with them (genie-ai-runtime §4, Path C:
// quants read as whole words and dequantised in registers).
//
// Activations.  Each 32-wide sub-block j of x is held as a 32-bit fixed-point
// integer X = rint(x / s_j) with a power-of-two scale s_j = 2^(e-30), e the
// exponent of the sub-block's largest |x| (so |X| <= 2^30), written in four
// balanced base-256 digits X = 2^24*D3 + 2^16*D2 + 2^8*D1 + D0, every digit a
// signed byte in [-128, 127].  The 4-bit quants q enter dp4a dot products with
// the digit planes unchanged, so each plane sum sum(q*D) is an exact integer
// of magnitude <= 15*128*32, and so is every pair 256*P_hi + P_lo of them; a
// sub-block's value is then formed with a single fp32 rounding:
//     tier 1:  P/256 ~ fmaf(256*P3 + P2, 256, P1)            (D0 dropped)
//     tier 2:  P/256 = fmaf(256*P3 + P2, 256, (256*P1 + P0)/256)
// and the scales are applied in fp32 registers:
//     acc += d*sc_j*s'_j*V_j - dmin*m_j*XS_j,   s'_j = 256*s_j, XS_j = sum x.
// Balanced digits keep every plane sum within twice sum q|X|, so combining
// the planes never cancels more than that.
//
// Tiers (chosen per sub-block when x is staged; all lanes of a warp read the
// same activations, so a tier is a warp-uniform branch):
//  - tier 1 (three planes D3..D1): every element keeps |x - s'*X'| <= 2^-14 |x|;
//  - tier 2 (all four planes): some element would not, but every nonzero
//    element keeps |x - s*X| <= 2^-14 |x| (a wide range inside the block);
//    D0 is added as a second exact integer term of the same rounding;
//  - tier 3 (fp32): any other block -- an element below ~2^-16 of the
//    block's largest, or a largest |x| outside [2^-87, 2^94) -- is staged
//    with scale 0 (and its fp32 activations in a small pool) and takes
//    V_j = sum q*x by fp32 multiply-adds after the integer loop.
// Tier-2 sub-blocks keep their D0 plane in a small per-warp pool of shared
// memory; a chunk holding one takes one extra warp-uniform branch.  A 32-bit
// word of quants (8 weights) costs a shift, two LOP3s and six dp4a per token
// (plus two dp4a in a tier-2 sub-block), against one fp32 multiply-add per
// weight for a dequantised dot.
#pragma once

#include "q4k_internal.h"
#include "tc_ptx.cuh"

#include <cuda_fp16.h>
#include <cstdint>

namespace q4k {
namespace gemv {

constexpr int kRegion = 208;     // bytes per (token, superblock, chunk) of the planes D3..D1: 192 + pad
constexpr int kStageWarps = 15;  // warps that stage x (the consumer warps of both kernels)
constexpr int kPool3PerWarp = 1; // fp32 activations of tier-3 sub-blocks a warp keeps (128 bytes each)
constexpr uint32_t kNoSlot = 0x3FFFu;   // a tier-3 sub-block without a pool slot reads x from global memory
// biased fp32 exponents of a sub-block's largest |x| staged in fixed point
constexpr int kEFixedMin = 40;    // 2^-87
constexpr int kEFixedMax = 220;   // below 2^94

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

// Shared-memory bytes of the staged activations: the planes D3..D1 (xs),
// then (xss) the (scale, sum) pair and the tag of every sub-block, the D0
// pool (per warp: pool2_per_warp slots of 32 bytes) and the tier-3 pool (per
// warp: kPool3PerWarp slots of 128 bytes).  Laid out for the nb being staged.
__host__ __device__ constexpr int pool2_per_warp(int B, int nb) {
  // about a quarter of a warp's sub-blocks; N(0,1) activations need ~9 %
  return (B * nb * 8 + 59) / 60 < 2 ? 2 : ((B * nb * 8 + 59) / 60 > 16 ? 16 : (B * nb * 8 + 59) / 60);
}
__host__ __device__ constexpr size_t tag_offset(int B, int nb) { return sizeof(float2) * (size_t)B * nb * 8; }
__host__ __device__ constexpr size_t pool2_offset(int B, int nb) {
  return (tag_offset(B, nb) + sizeof(uint16_t) * (size_t)B * nb * 8 + 15) & ~size_t(15);
}
__host__ __device__ constexpr size_t pool3_offset(int B, int nb) {
  return pool2_offset(B, nb) + 32 * (size_t)kStageWarps * pool2_per_warp(B, nb);
}
__host__ __device__ constexpr size_t xs_bytes(int B, int nb) { return (size_t)B * nb * 4 * kRegion; }
__host__ __device__ constexpr size_t xss_bytes(int B, int nb) {
  return pool3_offset(B, nb) + 128 * (size_t)kStageWarps * kPool3PerWarp;
}

// Staged activations as the consumers read them.
struct XView {
  const uint8_t* planes;   // [B][nb][4 chunks][kRegion]: planes D3..D1
  const float2* ss;        // [B][nb][8]: (scale s', fp32 sum of x); s' = 0 in tier 3
  const uint16_t* tag;     // [B][nb][8]: bits 0-1 tier-1 (0), -2 (1) or -3 (2); bits 2.. pool slot
  const uint8_t* pool2;    // [slot][32]: the D0 plane of a tier-2 sub-block
  const float* pool3;      // [slot][32]: the activations of a tier-3 sub-block
  const float* x;          // the activations themselves, [B][nb*256] (tier 3 without a slot)
  int nb;
};

__device__ __forceinline__ XView make_view(const uint8_t* xs, const float2* xss, const float* x, int B, int nb) {
  const uint8_t* base = reinterpret_cast<const uint8_t*>(xss);
  XView v;
  v.planes = xs;
  v.ss = xss;
  v.tag = reinterpret_cast<const uint16_t*>(base + tag_offset(B, nb));
  v.pool2 = base + pool2_offset(B, nb);
  v.pool3 = reinterpret_cast<const float*>(base + pool3_offset(B, nb));
  v.x = x;
  v.nb = nb;
  return v;
}

// byte k (0..3) of each of four words, gathered into one word
__device__ __forceinline__ uint32_t gather_byte(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int k) {
  const uint32_t sel = (uint32_t)k | ((uint32_t)(k + 4) << 4);
  return __byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410);
}

// Stage x [B][nb*256] once per CTA as balanced-digit planes of 32-bit fixed
// point, with each sub-block's scale, fp32 sum and tier.  Eight lanes hold
// one sub-block (four elements each), so its max and sum are three shuffles
// and its tier one ballot; all loads of a round are issued before any use.
// NT = 32 * kStageWarps threads (tid < NT) take part.  Each warp hands out
// the pool slots of the sub-blocks it stages from its own share of the
// pools, counting in registers (two ballots per round, no atomics); a tier-2 sub-block that finds the warp's share full goes to
// tier 3, and a tier-3 one without a slot reads x from global memory.
// kCoherent reads x through L2 only (x may have been written earlier in the
// same kernel); otherwise through the read-only path.
// Plane layout per (token, superblock, chunk c): 16-byte words at
// ((h*3 + p)*2 + s)*16, h = half of the chunk's 32 positions, p = plane
// (0, 1, 2 = digits D1, D2, D3), s = sub-block 2c (0) or 2c+1 (1); word k of
// it holds positions 16h+4k..+3.  A D0 pool slot (32 bytes) holds positions
// 4k..4k+3 in word k.
template <int B, int NT, bool kCoherent>
__device__ __forceinline__ void stage_x(const float* __restrict__ x, int nb, uint8_t* xs, float2* xss,
                                        int tid) {
  static_assert(NT == 32 * kStageWarps, "pools are laid out per staging warp");
  uint8_t* xb = reinterpret_cast<uint8_t*>(xss);
  uint16_t* tag = reinterpret_cast<uint16_t*>(xb + tag_offset(B, nb));
  uint32_t* pool2 = reinterpret_cast<uint32_t*>(xb + pool2_offset(B, nb));
  float4* pool3 = reinterpret_cast<float4*>(xb + pool3_offset(B, nb));
  const int lane = tid & 31, warp = tid >> 5;
  const int cap2 = pool2_per_warp(B, nb);
  int used2 = 0, used3 = 0;                          // warp-uniform
  const int row4 = nb * 64;                          // float4 per activation row
  const int n4 = B * row4;                           // a multiple of 64: whole warps
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
        // amax, so X = rint(x * 2^(156-E)) satisfies |X| <= 2^30
        const int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
        const bool fixed = E >= kEFixedMin && E <= kEFixedMax;
        const float mul = fixed ? __uint_as_float((uint32_t)(283 - E) << 23) : 0.0f;
        const float s24 = fixed ? __uint_as_float((uint32_t)(E - 21) << 23) : 0.0f;   // 2^(E-148)
        const float xv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t dg[4];
        bool t2 = false, t3 = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int X = __float2int_rn(xv[i] * mul);
          // balanced base-256 digits, each as a signed byte
          dg[i] = ((uint32_t)X + 0x80808080u) ^ 0x80808080u;
          const int ax = abs(X), d0 = abs((int)(int8_t)(dg[i] & 0xFFu));
          const bool nz = xv[i] != 0.0f;
          const bool e3 = nz && (!fixed || ax < (1 << 13));
          t3 = t3 || e3;
          t2 = t2 || e3 || (nz && ((d0 + 1) << 14) > ax);
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(xs + (((size_t)b * nb + sb) * 4 + c) * kRegion) +
                        (h * 3 * 2 + sf) * 4 + kw;
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) dst[pl * 2 * 4] = gather_byte(dg[0], dg[1], dg[2], dg[3], pl + 1);
        // a sub-block's tier: any of its eight lanes.  From the two ballots
        // every lane derives the warp's four groups' tiers, so the pool slots
        // (in group order) need no further exchange.
        const unsigned b2 = __ballot_sync(0xffffffffu, t2), b3 = __ballot_sync(0xffffffffu, t3);
        const int grp = lane & 24;
        unsigned want2 = 0u, want3 = 0u;   // bit g: group g takes a slot of the pool
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const bool g3g = ((b3 >> (8 * g)) & 0xFFu) != 0, g2g = !g3g && ((b2 >> (8 * g)) & 0xFFu) != 0;
          want2 |= (g2g ? 1u : 0u) << g;
          want3 |= (g3g ? 1u : 0u) << g;
        }
        const int gi = grp >> 3;
        const unsigned before = (1u << gi) - 1u;
        const bool g2 = (want2 >> gi) & 1u;
        const int slot2 = used2 + __popc(want2 & before);
        const bool in2 = g2 && slot2 < cap2;
        // tier-2 groups beyond the warp's share of the pool go to tier 3
        unsigned over = 0u;
        {
          int k = used2;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if ((want2 >> g) & 1u) {
              if (k >= cap2) over |= 1u << g;
              ++k;
            }
        }
        used2 += __popc(want2);
        want3 |= over;
        const bool g3 = (want3 >> gi) & 1u;
        const int slot3 = used3 + __popc(want3 & before);
        used3 += __popc(want3);
        const bool in3 = g3 && slot3 < kPool3PerWarp;
        const int s2 = warp * cap2 + slot2, s3 = warp * kPool3PerWarp + slot3;
        if (in2) pool2[(size_t)s2 * 8 + (pos >> 2)] = gather_byte(dg[0], dg[1], dg[2], dg[3], 0);
        if (in3) pool3[(size_t)s3 * 8 + (pos >> 2)] = v[u];
        if ((idx & 7) == 0) {
          const size_t e = ((size_t)b * nb + sb) * 8 + j;
          xss[e] = make_float2(g3 ? 0.0f : s24, sum);
          tag[e] = (uint16_t)(g3 ? 2u | ((in3 ? (uint32_t)s3 : kNoSlot) << 2) : (in2 ? 1u | ((uint32_t)s2 << 2) : 0u));
        }
      }
    }
  }
}

// fp32 dot of the 32 quants of sub-block j of the BLOCK144 superblock at
// `p` (shared memory) with its activations (the tier-3 path): xs[0..31] in
// shared memory, or, without a pool slot, xg[0..31] in global memory
template <bool kCoherent>
__device__ __forceinline__ float subblock_fp32(const uint8_t* p, int j, const float* xs, const float* xg) {
  const uint8_t* qs = p + 16 + 32 * (j >> 1);
  const int sh = (j & 1) ? 4 : 0;
  float v = 0.0f;
  if (xs) {
#pragma unroll 8
    for (int l = 0; l < 32; ++l) v = fmaf((float)((qs[l] >> sh) & 15), xs[l], v);
  } else {
#pragma unroll 8
    for (int l = 0; l < 32; ++l) {
      const float xl = kCoherent ? __ldcg(xg + l) : __ldg(xg + l);
      v = fmaf((float)((qs[l] >> sh) & 15), xl, v);
    }
  }
  return v;
}

// What the tier-3 sub-blocks among chunks c0 .. c0+cpl-1 add to the lane's
// scaled sum for token b: sc_j * sum q*x in fp32 (they were staged with scale
// 0, so the planes added nothing).  Out of line: rare, and the main loop
// keeps its registers.
template <bool kCoherent>
__device__ __noinline__ float tier3_fix(const uint8_t* p, const XView X, int sb, int c0, int cpl, int b,
                                        uint32_t sc03, uint32_t sc47) {
  const int nb = X.nb;
  const uint16_t* tg = X.tag + ((size_t)b * nb + sb) * 8;
  float add = 0.0f;
  for (int j = 2 * c0; j < 2 * (c0 + cpl); ++j) {
    const uint32_t t = tg[j];
    if (!(t & 2u)) continue;
    const float sc = byte_f(j < 4 ? sc03 : sc47, j & 3);
    const float* xg = X.x + (size_t)b * nb * 256 + (size_t)sb * 256 + 32 * j;
    const float* xs = (t >> 2) != kNoSlot ? X.pool3 + 32 * (size_t)(t >> 2) : nullptr;
    add = fmaf(sc, subblock_fp32<kCoherent>(p, j, xs, xg), add);
  }
  return add;
}

// One lane's share of one superblock row against the staged activations:
// chunks c0 .. c0+CPL-1 (64 weights each) of the BLOCK144 superblock at `p`
// (shared memory), superblock index sb of x.  acc[b] receives
// d * sum_j sc_j s'_j V_j - dmin * sum_j m_j XS_j over the lane's sub-blocks.
// Per chunk the three planes D3..D1 of both sub-blocks, then, only where a
// sub-block is in tier 2, its D0 plane; tier-3 sub-blocks are added after.
template <int B, int CPL, bool kCoherent>
__device__ __forceinline__ void superblock_dot(const uint8_t* p, const XView& X, int sb, int c0,
                                               float (&acc)[B]) {
  const int nb = X.nb;
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
    // exact integer sums of q * D per digit plane D1..D3, low (sub-block 2c)
    // and high (2c+1) nibbles
    int lo[B][3], hi[B][3];
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
      for (int pl = 0; pl < 3; ++pl) lo[b][pl] = hi[b][pl] = 0;
    const uint8_t* xc0 = X.planes + ((size_t)sb * 4 + c) * kRegion;
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
            lo[b][pl] = dp4a_us(ql[k], word_of(xl, k), lo[b][pl]);
            hi[b][pl] = dp4a_us(qh[k], word_of(xh, k), hi[b][pl]);
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
      // tier 2: the D0 planes of the chunk's flagged sub-blocks, from the pool
      const uint32_t tw = *reinterpret_cast<const uint32_t*>(X.tag + ((size_t)b * nb + sb) * 8 + 2 * c);
      int p0_lo = 0, p0_hi = 0;
      if (tw & 0x00010001u) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 qq = h ? q1 : q0;
          if ((tw & 3u) == 1u) {
            const uint4 xw = reinterpret_cast<const uint4*>(X.pool2 + 32 * (size_t)((tw >> 2) & 0x3FFFu))[h];
#pragma unroll
            for (int k = 0; k < 4; ++k) p0_lo = dp4a_us(word_of(qq, k) & 0x0F0F0F0Fu, word_of(xw, k), p0_lo);
          }
          if (((tw >> 16) & 3u) == 1u) {
            const uint4 xw = reinterpret_cast<const uint4*>(X.pool2 + 32 * (size_t)(tw >> 18))[h];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              p0_hi = dp4a_us((word_of(qq, k) >> 4) & 0x0F0F0F0Fu, word_of(xw, k), p0_hi);
          }
        }
      }
      // P/256 in units of s' = 256 s, one rounding (exact integer parts;
      // without tier 2, p0 = 0 and the second term is the integer P1)
      const float v_lo = fmaf((float)(lo[b][2] * 256 + lo[b][1]), 256.0f, (float)(lo[b][0] * 256 + p0_lo) * 0.00390625f);
      const float v_hi = fmaf((float)(hi[b][2] * 256 + hi[b][1]), 256.0f, (float)(hi[b][0] * 256 + p0_hi) * 0.00390625f);
      const float4 ss = *reinterpret_cast<const float4*>(X.ss + ((size_t)b * nb + sb) * 8 + 2 * c);
      scaled[b] = fmaf(sc_hi * ss.z, v_hi, fmaf(sc_lo * ss.x, v_lo, scaled[b]));
      mins[b] = fmaf(m_hi, ss.w, fmaf(m_lo, ss.y, mins[b]));
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = fmaf(dm.x, scaled[b], -dm.y * mins[b]);
  // tier-3 sub-blocks among the lane's chunks (rare)
#pragma unroll
  for (int b = 0; b < B; ++b) {
    // the tags of the lane's sub-blocks 2c0 .. 2(c0+CPL)-1, two per word
    const uint4 t8 = *reinterpret_cast<const uint4*>(X.tag + ((size_t)b * nb + sb) * 8);
    uint32_t any;
    if (CPL == 4) any = t8.x | t8.y | t8.z | t8.w;
    else if (CPL == 2) any = c0 ? (t8.z | t8.w) : (t8.x | t8.y);
    else any = word_of(t8, c0);
    if (any & 0x00020002u) acc[b] = fmaf(dm.x, tier3_fix<kCoherent>(p, X, sb, c0, CPL, b, sc03, sc47), acc[b]);
  }
}

// ---------------------------------------------------------------------------
// q8_1 activations (the MMQ form for a few tokens).  The int8 quants of one
// (token, superblock, chunk) take one 64-byte region laid out like a digit
// plane: 16-byte words at (h*2 + s)*16, word k holding positions
// 16h+4k..+3 of sub-block 2c+s.  Per sub-block: (d8, d8*S) as a float2.
constexpr int kRegionQ8 = 64;
__host__ __device__ constexpr size_t xq8_bytes(int B, int nb) { return (size_t)B * nb * 4 * kRegionQ8; }
__host__ __device__ constexpr size_t xq8s_bytes(int B, int nb) { return sizeof(float2) * (size_t)B * nb * 8; }

// Stage q8 [B][nb*256] (int8, or binary16 integers when kH16), d8 and the
// block sums once per CTA.  One thread takes 16 quants (half a sub-block).
template <int B, int NT, bool kH16>
__device__ __forceinline__ void stage_q8(const void* __restrict__ q8, const float* __restrict__ d8,
                                         const int32_t* __restrict__ ssum, int nb, uint8_t* xs, float2* xss,
                                         int tid) {
  const int n16 = B * nb * 16;   // halves of sub-blocks
  for (int i = tid; i < n16; i += NT) {
    const int b = i / (nb * 16), rem = i - b * nb * 16;
    const int sb = rem >> 4, j = (rem >> 1) & 7, h = rem & 1;
    const int c = j >> 1, sf = j & 1;
    const size_t e0 = ((size_t)b * nb + sb) * 256 + 32 * j + 16 * h;   // first element
    uint4 w;
    if (kH16) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q8) + e0);
      const uint4 a = __ldg(src), bq = __ldg(src + 1);
      const uint32_t hw[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
      uint32_t out[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 lo = *reinterpret_cast<const __half2*>(&hw[2 * k]);
        const __half2 hi = *reinterpret_cast<const __half2*>(&hw[2 * k + 1]);
        const int v0 = __half2int_rn(__low2half(lo)), v1 = __half2int_rn(__high2half(lo));
        const int v2 = __half2int_rn(__low2half(hi)), v3 = __half2int_rn(__high2half(hi));
        out[k] = (uint32_t)(v0 & 0xFF) | ((uint32_t)(v1 & 0xFF) << 8) | ((uint32_t)(v2 & 0xFF) << 16) |
                 ((uint32_t)(v3 & 0xFF) << 24);
      }
      w = make_uint4(out[0], out[1], out[2], out[3]);
    } else {
      w = __ldg(reinterpret_cast<const uint4*>(static_cast<const int8_t*>(q8) + e0));
    }
    *reinterpret_cast<uint4*>(xs + (((size_t)b * nb + sb) * 4 + c) * kRegionQ8 + (h * 2 + sf) * 16) = w;
    if (h == 0) {   // (scales are absent when only the block dots are wanted)
      const size_t sbk = ((size_t)b * nb + sb) * 8 + j;
      const float dd = d8 ? __ldg(d8 + sbk) : 0.0f;
      xss[sbk] = make_float2(dd, ssum ? dd * (float)__ldg(ssum + sbk) : 0.0f);
    }
  }
}

// superblock_dot for q8 activations: per sub-block the exact integer
// P = sum q*q8 (dp4a, |P| <= 15*127*32), then
//     acc += d*sc_j*d8_j*P_j - dmin*m_j*(d8_j*S_j).
// With `pout` (test export) each P_j is stored at pout[b * pstride + j]
// (the lane's sub-blocks only).
template <int B, int CPL>
__device__ __forceinline__ void superblock_dot_q8(const uint8_t* p, const uint8_t* xs, const float2* xss, int nb,
                                                  int sb, int c0, float (&acc)[B], int32_t* pout, size_t pstride) {
  const uint4 hd = *reinterpret_cast<const uint4*>(p);
  const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
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
    int lo[B], hi[B];
#pragma unroll
    for (int b = 0; b < B; ++b) lo[b] = hi[b] = 0;
    const uint8_t* xc0 = xs + ((size_t)sb * 4 + c) * kRegionQ8;
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
        const uint4* xp = reinterpret_cast<const uint4*>(xc0 + (size_t)b * nb * 4 * kRegionQ8) + h * 2;
        const uint4 xl = xp[0], xh = xp[1];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo[b] = dp4a_us(ql[k], word_of(xl, k), lo[b]);
          hi[b] = dp4a_us(qh[k], word_of(xh, k), hi[b]);
        }
      }
    }
    const uint32_t scw = c < 2 ? sc03 : sc47, mw = c < 2 ? m03 : m47;
    const int bi = 2 * (c & 1);
    const float sc_lo = byte_f(scw, bi), sc_hi = byte_f(scw, bi + 1);
    const float m_lo = byte_f(mw, bi), m_hi = byte_f(mw, bi + 1);
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float4 ss = *reinterpret_cast<const float4*>(xss + ((size_t)b * nb + sb) * 8 + 2 * c);
      scaled[b] = fmaf(sc_hi * ss.z, (float)hi[b], fmaf(sc_lo * ss.x, (float)lo[b], scaled[b]));
      mins[b] = fmaf(m_hi, ss.w, fmaf(m_lo, ss.y, mins[b]));
      if (pout) {
        pout[(size_t)b * pstride + 2 * c] = lo[b];
        pout[(size_t)b * pstride + 2 * c + 1] = hi[b];
      }
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = fmaf(dm.x, scaled[b], -dm.y * mins[b]);
}

// ---------------------------------------------------------------------------
// Q6_K superblocks in the GPU layout (q6k_pack.cu): 16 int8 scales, then four
// 48-byte chunks of 64 weights -- 32 bytes of low nibbles (sub-block s = 0 in
// the low nibble, s = 1 in the high, as in BLOCK144) and 16 bytes of high bit
// pairs, pair f = 2s + h of byte i for position 16h + i of sub-block s, its
// upper bit inverted.  The quant word for positions 16h+4k..+3 of sub-block s
// is assembled as the signed bytes 4*(q - 32): the low nibble shifted to bits
// 2-5 and the bit pair to bits 6-7, where the inverted pair reads as the
// signed value hi - 2.  Each 16-weight scale group then takes the exact
// integer 4*P per digit plane from four dp4a (|4P| <= 16*128*128).
constexpr int kQ6Blk = 208;   // bytes of a GPU-layout Q6_K superblock

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int acc) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(acc));
  return d;
}

// signed bytes 4*(q - 32) of sub-block s, half h, word k: l = low-nibble
// word (h, k), hw = high-pair word k of the chunk
__device__ __forceinline__ uint32_t q6_word(uint32_t l, uint32_t hw, int s, int h) {
  const uint32_t lo = (s ? (l >> 2) : (l << 2)) & 0x3C3C3C3Cu;
  const int f = 2 * s + h;
  return ((hw << (6 - 2 * f)) & 0xC0C0C0C0u) | lo;
}

// sum over the 32 weights of sub-block j (0..7) of the Q6_K superblock at p
// of sc_g * (q - 32) * x, in fp32 (the tier-3 path); activations as in
// subblock_fp32
template <bool kCoherent>
__device__ __forceinline__ float subblock_fp32_q6(const uint8_t* p, int j, const float* xs, const float* xg) {
  const uint8_t* ch = p + 16 + 48 * (j >> 1);
  const int s = j & 1;
  float v = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float part = 0.0f;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int t = 16 * h + i;
      const int lo = (ch[t] >> (4 * s)) & 15;
      const int hi = (int)(((ch[32 + i] >> (2 * (2 * s + h))) & 3u) ^ 2u);
      const float xl = xs ? xs[t] : (kCoherent ? __ldcg(xg + t) : __ldg(xg + t));
      part = fmaf((float)(lo + 16 * hi - 32), xl, part);
    }
    v = fmaf((float)(int8_t)p[2 * j + h], part, v);
  }
  return v;
}

template <bool kCoherent>
__device__ __noinline__ float tier3_fix_q6(const uint8_t* p, const XView X, int sb, int c0, int cpl, int b) {
  const int nb = X.nb;
  const uint16_t* tg = X.tag + ((size_t)b * nb + sb) * 8;
  float add = 0.0f;
  for (int j = 2 * c0; j < 2 * (c0 + cpl); ++j) {
    const uint32_t t = tg[j];
    if (!(t & 2u)) continue;
    const float* xg = X.x + (size_t)b * nb * 256 + (size_t)sb * 256 + 32 * j;
    const float* xs = (t >> 2) != kNoSlot ? X.pool3 + 32 * (size_t)(t >> 2) : nullptr;
    add += subblock_fp32_q6<kCoherent>(p, j, xs, xg);
  }
  return add;
}

// superblock_dot for a Q6_K superblock (GPU layout, shared memory) with scale
// d: acc[b] = d * sum_g sc_g s'_g V_g over the lane's chunks c0 .. c0+CPL-1,
// V_g the group's P/256 in units of s' = 256 s (one rounding, as for Q4_K;
// the factor 4 of the quant bytes is taken out by the combine's constants).
// Tier-2 and tier-3 sub-blocks as in superblock_dot.
template <int B, int CPL, bool kCoherent>
__device__ __forceinline__ void superblock_dot_q6(const uint8_t* p, float d, const XView& X, int sb, int c0,
                                                  float (&acc)[B]) {
  const int nb = X.nb;
  const uint4 scv = *reinterpret_cast<const uint4*>(p);   // int8 scales of groups 0..15
  float scaled[B];
#pragma unroll
  for (int b = 0; b < B; ++b) scaled[b] = 0.0f;
#pragma unroll
  for (int cc = 0; cc < CPL; ++cc) {
    const int c = c0 + cc;
    const uint8_t* ch = p + 16 + 48 * c;
    const uint4 hwv = *reinterpret_cast<const uint4*>(ch + 32);
    const uint32_t scw = word_of(scv, c);   // groups 4c + 2s + h
    const uint8_t* xc0 = X.planes + ((size_t)sb * 4 + c) * kRegion;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 lv = *reinterpret_cast<const uint4*>(ch + 16 * h);
      uint32_t w0[4], w1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w0[k] = q6_word(word_of(lv, k), word_of(hwv, k), 0, h);
        w1[k] = q6_word(word_of(lv, k), word_of(hwv, k), 1, h);
      }
      const float sc0 = (float)(int8_t)((scw >> (8 * h)) & 0xFFu);
      const float sc1 = (float)(int8_t)((scw >> (8 * (2 + h))) & 0xFFu);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint4* xp = reinterpret_cast<const uint4*>(xc0 + (size_t)b * nb * 4 * kRegion) + h * 6;
        int a0[3], a1[3];
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
          const uint4 xl = xp[2 * pl], xh = xp[2 * pl + 1];
          a0[pl] = a1[pl] = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            a0[pl] = dp4a_ss(w0[k], word_of(xl, k), a0[pl]);
            a1[pl] = dp4a_ss(w1[k], word_of(xh, k), a1[pl]);
          }
        }
        const uint32_t tw = *reinterpret_cast<const uint32_t*>(X.tag + ((size_t)b * nb + sb) * 8 + 2 * c);
        int p00 = 0, p01 = 0;
        if (tw & 0x00010001u) {
          if ((tw & 3u) == 1u) {
            const uint4 xw = reinterpret_cast<const uint4*>(X.pool2 + 32 * (size_t)((tw >> 2) & 0x3FFFu))[h];
#pragma unroll
            for (int k = 0; k < 4; ++k) p00 = dp4a_ss(w0[k], word_of(xw, k), p00);
          }
          if (((tw >> 16) & 3u) == 1u) {
            const uint4 xw = reinterpret_cast<const uint4*>(X.pool2 + 32 * (size_t)(tw >> 18))[h];
#pragma unroll
            for (int k = 0; k < 4; ++k) p01 = dp4a_ss(w1[k], word_of(xw, k), p01);
          }
        }
        // (4P)/1024 = P/256 in units of s'
        const float v0 = fmaf((float)(a0[2] * 256 + a0[1]), 64.0f, (float)(a0[0] * 256 + p00) * 0.0009765625f);
        const float v1 = fmaf((float)(a1[2] * 256 + a1[1]), 64.0f, (float)(a1[0] * 256 + p01) * 0.0009765625f);
        const float4 ss = *reinterpret_cast<const float4*>(X.ss + ((size_t)b * nb + sb) * 8 + 2 * c);
        scaled[b] = fmaf(sc1 * ss.z, v1, fmaf(sc0 * ss.x, v0, scaled[b]));
      }
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = d * scaled[b];
#pragma unroll
  for (int b = 0; b < B; ++b) {
    const uint4 t8 = *reinterpret_cast<const uint4*>(X.tag + ((size_t)b * nb + sb) * 8);
    uint32_t any;
    if (CPL == 4) any = t8.x | t8.y | t8.z | t8.w;
    else if (CPL == 2) any = c0 ? (t8.z | t8.w) : (t8.x | t8.y);
    else any = word_of(t8, c0);
    if (any & 0x00020002u) acc[b] = fmaf(d, tier3_fix_q6<kCoherent>(p, X, sb, c0, CPL, b), acc[b]);
  }
}

// superblock_dot_q6 for q8_1 activations (the MMQ form): per 16-weight
// group g the exact integer P_g = sum (q - 32) * q8 (dp4a on the 4*(q-32)
// words, then /4), and acc[b] = d * sum_g sc_g * d8_(g/2) * P_g.  With
// `pout` (test export) each P_g is stored at pout[b * pstride + g] (the
// lane's groups only).
template <int B, int CPL>
__device__ __forceinline__ void superblock_dot_q6_q8(const uint8_t* p, float d, const uint8_t* xs,
                                                     const float2* xss, int nb, int sb, int c0, float (&acc)[B],
                                                     int32_t* pout, size_t pstride) {
  const uint4 scv = *reinterpret_cast<const uint4*>(p);
  float scaled[B];
#pragma unroll
  for (int b = 0; b < B; ++b) scaled[b] = 0.0f;
#pragma unroll
  for (int cc = 0; cc < CPL; ++cc) {
    const int c = c0 + cc;
    const uint8_t* ch = p + 16 + 48 * c;
    const uint4 hwv = *reinterpret_cast<const uint4*>(ch + 32);
    const uint32_t scw = word_of(scv, c);
    const uint8_t* xc0 = xs + ((size_t)sb * 4 + c) * kRegionQ8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 lv = *reinterpret_cast<const uint4*>(ch + 16 * h);
      uint32_t w0[4], w1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w0[k] = q6_word(word_of(lv, k), word_of(hwv, k), 0, h);
        w1[k] = q6_word(word_of(lv, k), word_of(hwv, k), 1, h);
      }
      const float sc0 = (float)(int8_t)((scw >> (8 * h)) & 0xFFu);
      const float sc1 = (float)(int8_t)((scw >> (8 * (2 + h))) & 0xFFu);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint4* xp = reinterpret_cast<const uint4*>(xc0 + (size_t)b * nb * 4 * kRegionQ8) + h * 2;
        const uint4 xl = xp[0], xh = xp[1];
        int a0 = 0, a1 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a0 = dp4a_ss(w0[k], word_of(xl, k), a0);
          a1 = dp4a_ss(w1[k], word_of(xh, k), a1);
        }
        const int p0 = a0 / 4, p1 = a1 / 4;   // exact: every product is a multiple of 4
        const float4 ss = *reinterpret_cast<const float4*>(xss + ((size_t)b * nb + sb) * 8 + 2 * c);
        scaled[b] = fmaf(sc1 * ss.z, (float)p1, fmaf(sc0 * ss.x, (float)p0, scaled[b]));
        if (pout) {
          pout[(size_t)b * pstride + 4 * c + h] = p0;
          pout[(size_t)b * pstride + 4 * c + 2 + h] = p1;
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = d * scaled[b];
}

}  // namespace gemv
}  // namespace q4k
