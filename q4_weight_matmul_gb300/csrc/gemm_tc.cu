// q4k_gemm on the sm_103a tensor cores: the prefill MMQ GEMM over q8_1
// activations (genie-ai-runtime §3, "The tensor-core kernel (Path E)" is the
// prior art; this is the integer MMQ form of it).
//
//   y[t][o] = sum_b d*sc[o,b] * d8[t,b] * P[t,o,b] - dmin*m[o,b] * d8[t,b] * S[t,b]
//   P[t,o,b] = sum_{i<32} q[o][32b+i] * q8[t][32b+i]
//
// sm_103a has no integer tcgen05 MMA, so the integer dots run on kind::f16
// with operands that are exact small integers: A = q8 (|q8| <= 127) and
// B = sc*q (<= 63*15 = 945), both exact in fp16.  Every product and every
// partial sum of one 32-wide block (|sum| <= 945*127*32 < 2^22) is an integer
// that fp32 holds exactly, so the fp32 TMEM accumulator of a block equals
// sc*P exactly, whatever order the tensor core adds in.
//
// Tile: 128 tokens (TMEM lanes) x 128 weight rows (TMEM columns); K walks
// 64 weights per pipeline stage.  Warp roles in one CTA of 16 warps (four per
// SM sub-partition, so every thread may hold 128 registers):
//   warp 0      allocates TMEM; lane 0 issues every tcgen05.mma
//   warps 1-7   converters: read q8 and packed superblocks from global memory,
//               widen them to fp16 (B pre-multiplied by sc) and store them in
//               the 128-byte-swizzled K-major layout the MMA reads
//   warps 8-15  epilogue: per block, read the block's accumulator from TMEM
//               and add it, times the token's scale d8, into a per-superblock
//               sum; per superblock, add d * sum into a running fp32 total kept
//               in TMEM
// TMEM columns: [0,128) and [128,256) double-buffered block accumulators,
// [256,384) the min-term accumulator, [384,512) the running total.
//
// The min term sum_b (dmin*m[o,b]) * (d8*S[t,b]) is a depth-(K/32) product;
// it runs on the tensor cores too (bf16, both factors split into two bf16
// parts, 4 products per block, ~2^-16 relative error), one extra stage after
// every two superblocks, into its own accumulator.
//
// Every mbarrier wait is bounded (tc::kTimeoutNs); a wait that gives up sets
// the library's device error word, raises a CTA-wide abort flag and the CTA
// unwinds, drains its MMAs and frees its TMEM.
#include "q4k_internal.h"
#include "tc_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kBM = 128;                 // tokens per tile
constexpr int kBN = 128;                 // weight rows per tile
constexpr int kStages = 4;
constexpr int kTileBytes = 128 * 128;    // 128 rows x 64 k x fp16
constexpr int kConvWarps = 7;
constexpr int kEpiWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 32 * (1 + kConvWarps + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColMin = 256;
constexpr uint32_t kColAcc = 384;

struct __align__(1024) Smem {
  uint8_t a[kStages][kTileBytes];
  uint8_t b[kStages][kTileBytes];
  float dsm[2][kBN];
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[2], tempty[2];
  uint64_t dfull[2], dempty[2];
  uint64_t mfull, drain;
  uint32_t tmem_base;
  int abort;
};

struct StageInfo {
  int kind;   // 0: main (64 weights of one superblock), 1: min-term stage
  int sb;     // superblock (main) or first superblock of the pair (min)
  int c;      // 64-weight chunk of the superblock (main)
};

__device__ __forceinline__ StageInfo stage_info(int s, int nsb, bool with_min) {
  StageInfo si;
  if (!with_min) {
    si.kind = 0;
    si.sb = s >> 2;
    si.c = s & 3;
    return si;
  }
  const int p = s / 9, r = s - 9 * p;
  const int main_in_pair = 4 * min(2, nsb - 2 * p);
  if (r < main_in_pair) {
    si.kind = 0;
    si.sb = 2 * p + (r >> 2);
    si.c = r & 3;
  } else {
    si.kind = 1;
    si.sb = 2 * p;
    si.c = 0;
  }
  return si;
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four int8 (k0..k3) to fp16 pairs ordered (k0,k2), (k1,k3): bias each byte
// by 128, place it under the fp16 exponent of 1024 and subtract 1152.
__device__ __forceinline__ void s8x4_to_h2(uint32_t v, uint32_t& p02, uint32_t& p13) {
  const uint32_t u = v ^ 0x80808080u;
  const __half2 off = u2h(0x64806480u);   // (1152, 1152)
  p02 = h2u(__hsub2(u2h(prmt(u, 0x64646464u, 0x4240u)), off));
  p13 = h2u(__hsub2(u2h(prmt(u, 0x64646464u, 0x4341u)), off));
}

// One word of quant bytes (weights l..l+3 of the low sub-block in the low
// nibbles, of the high sub-block in the high nibbles) to sc*q fp16 pairs in
// the (l,l+2), (l+1,l+3) order.  Low nibbles sit under the exponent of 1024
// as 1024+q, high nibbles as 1024+16q; one exact FMA each removes the bias
// and applies the sub-block scale.
__device__ __forceinline__ void q4x8_to_h2(uint32_t w, __half2 m_lo, __half2 a_lo, __half2 m_hi,
                                           __half2 a_hi, uint32_t (&lo)[2], uint32_t (&hi)[2]) {
  const uint32_t w8 = w >> 8;
  lo[0] = h2u(__hfma2(u2h((w & 0x000F000Fu) | 0x64006400u), m_lo, a_lo));
  lo[1] = h2u(__hfma2(u2h((w8 & 0x000F000Fu) | 0x64006400u), m_lo, a_lo));
  hi[0] = h2u(__hfma2(u2h((w & 0x00F000F0u) | 0x64006400u), m_hi, a_hi));
  hi[1] = h2u(__hfma2(u2h((w8 & 0x00F000F0u) | 0x64006400u), m_hi, a_hi));
}

__device__ __forceinline__ void sts128(uint8_t* base, uint32_t off, uint32_t x, uint32_t y, uint32_t z,
                                       uint32_t w) {
  *reinterpret_cast<uint4*>(base + off) = make_uint4(x, y, z, w);
}

// scale (sc) and min (m) of sub-block j from a superblock header
__device__ __forceinline__ void scale_min(const uint4& h, int j, uint32_t& sc, uint32_t& m) {
  const uint32_t s03 = h.y, s47 = h.z, s811 = h.w;
  const int jj = j & 3;
  const uint32_t b1 = (s03 >> (8 * jj)) & 0xFFu, b2 = (s47 >> (8 * jj)) & 0xFFu,
                 b3 = (s811 >> (8 * jj)) & 0xFFu;
  if (j < 4) {
    sc = b1 & 63u;
    m = b2 & 63u;
  } else {
    sc = (b3 & 15u) | ((b1 >> 6) << 4);
    m = (b3 >> 4) | ((b2 >> 6) << 4);
  }
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// f = hi + lo with hi = bf16(f) and lo = bf16(f - hi)
__device__ __forceinline__ void split_bf16(float f, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(f));
  lo = __bfloat162float(__float2bfloat16_rn(f - hi));
}

// Raw global data of one stage for one converter thread.  Main stage:
// v[0..2] q8 runs of A units, v[3..4] quant bytes of B units, v[5..6] their
// rows' headers (first chunk of a superblock only).  Min stage: v[4u..4u+3]
// = d8 (two vectors) and block sums (two vectors) of unit u.
struct Raw {
  uint4 v[8];
};

// Work units of one stage: A units (token, 16-weight run) 512, B units
// (row, 16 quant bytes) 256; min stages use 256 (token|row, superblock) units.
constexpr int kUnitsA = 512;
constexpr int kUnitsB = 256;

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(
    const uint8_t* __restrict__ w, int rows, int nb, const int8_t* __restrict__ q8,
    const float* __restrict__ d8, const int32_t* __restrict__ ssum, int tokens,
    float* __restrict__ y, int32_t* __restrict__ p_out, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_flag = &sm.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kBN, tok0 = blockIdx.y * kBM;
  const int K = nb * kQK, nsub = K / kSub;
  const bool dots_only = p_out != nullptr;
  const bool with_min = !dots_only;
  const int n_stages = with_min ? 4 * nb + (nb + 1) / 2 : 4 * nb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&sm.full[i], kConvThreads);
      tc::mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.tfull[i], 1);
      tc::mbar_init(&sm.tempty[i], kEpiWarps);
      tc::mbar_init(&sm.dfull[i], kConvThreads);
      tc::mbar_init(&sm.dempty[i], kEpiWarps);
    }
    tc::mbar_init(&sm.mfull, 1);
    tc::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  auto fail = [&]() {
    if (!*abort_flag) atomicOr(err, 1);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idf = tc::idesc_f16(kBM, kBN, false);
      const uint32_t idb = tc::idesc_f16(kBM, kBN, true);
      int blk = 0, nmin = 0;
      bool ok = true;
      for (int s = 0; s < n_stages && ok; ++s) {
        const StageInfo si = stage_info(s, nb, with_min);
        const int st = s % kStages;
        if (!tc::mbar_wait(&sm.full[st], (s / kStages) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t a_base = tc::smem_u32(sm.a[st]), b_base = tc::smem_u32(sm.b[st]);
        if (si.kind == 0) {
          for (int h = 0; h < 2; ++h) {
            const int buf = blk & 1;
            if (!tc::mbar_wait(&sm.tempty[buf], ((blk >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t koff = (uint32_t)(2 * h + kk) * 32u;
              tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_base + koff),
                             tc::desc_sw128(b_base + koff), idf, (uint32_t)kk);
            }
            tc::mma_commit(&sm.tfull[buf]);
            ++blk;
          }
          if (!ok) break;
        } else {
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f16_ss(tmem + kColMin, tc::desc_sw128(a_base + 32u * kk),
                           tc::desc_sw128(b_base + 32u * kk), idb, (nmin > 0 || kk > 0) ? 1u : 0u);
          ++nmin;
        }
        tc::mma_commit(&sm.empty[st]);
      }
      if (!ok) fail();
      tc::mma_commit(&sm.mfull);
      // drain: every MMA issued above has completed before TMEM is freed
      tc::mma_commit(&sm.drain);
      int never = 0;
      if (!tc::mbar_wait(&sm.drain, 0, &never)) fail();
    }
  } else if (warp <= kConvWarps) {
    // ------------------------------------------------------------ converters
    const int ci = threadIdx.x - 32;
    uint4 hdr_keep[2][2];   // [B unit slot][superblock parity]
    for (int i = 0; i < 2; ++i) hdr_keep[i][0] = hdr_keep[i][1] = make_uint4(0, 0, 0, 0);

    auto load = [&](int s) {
      Raw r;
#pragma unroll
      for (int i = 0; i < 8; ++i) r.v[i] = make_uint4(0, 0, 0, 0);
      const StageInfo si = stage_info(s, nb, with_min);
      if (si.kind == 0) {
#pragma unroll
        for (int ua = 0; ua < 3; ++ua) {
          const int u = ci + kConvThreads * ua;
          if (u < kUnitsA) {
            const int tok = tok0 + (u >> 2);
            if (tok < tokens) r.v[ua] = ldg16(q8 + (size_t)tok * K + kQK * si.sb + 64 * si.c + 16 * (u & 3));
          }
        }
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) {
          const int u = ci + kConvThreads * ub;
          const int row = row0 + (u >> 1);
          if (u < kUnitsB && row < rows) {
            const uint8_t* sbp = w + ((size_t)row * nb + si.sb) * kBlockBytes;
            r.v[3 + ub] = ldg16(sbp + 16 + 32 * si.c + 16 * (u & 1));
            if (si.c == 0) r.v[5 + ub] = ldg16(sbp);
          }
        }
      } else {
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) {
          const int u = ci + kConvThreads * ub;
          const int tok = tok0 + (u >> 1), sbm = si.sb + (u & 1);
          if (u < kUnitsB && tok < tokens && sbm < nb) {
            const size_t off = (size_t)tok * nsub + 8 * sbm;
            r.v[4 * ub + 0] = ldg16(d8 + off);
            r.v[4 * ub + 1] = ldg16(d8 + off + 4);
            r.v[4 * ub + 2] = ldg16(ssum + off);
            r.v[4 * ub + 3] = ldg16(ssum + off + 4);
          }
        }
      }
      return r;
    };

    Raw cur = load(0);
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      Raw nxt;
      if (s + 1 < n_stages) nxt = load(s + 1);
      const StageInfo si = stage_info(s, nb, with_min);
      const int st = s % kStages;
      if (si.kind == 0 && si.c == 0) {
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) hdr_keep[ub][si.sb & 1] = cur.v[5 + ub];
        if (!tc::mbar_wait(&sm.dempty[si.sb & 1], ((si.sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) {
          const int u = ci + kConvThreads * ub;
          if (u < kUnitsB && (u & 1) == 0)
            sm.dsm[si.sb & 1][u >> 1] =
                __half2float(__ushort_as_half((unsigned short)(cur.v[5 + ub].x & 0xFFFFu)));
        }
        tc::mbar_arrive(&sm.dfull[si.sb & 1]);
      }
      if (!tc::mbar_wait(&sm.empty[st], ((s / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
      uint8_t* at = sm.a[st];
      uint8_t* bt = sm.b[st];
      if (si.kind == 0) {
        // A: a run of 16 int8 -> two 16-byte fp16 chunks
#pragma unroll
        for (int ua = 0; ua < 3; ++ua) {
          const int u = ci + kConvThreads * ua;
          if (u < kUnitsA) {
            const int ar = u >> 2, aq = u & 3;
            const uint4 v = cur.v[ua];
            uint32_t c0, c1, c2, c3, c4, c5, c6, c7;
            s8x4_to_h2(v.x, c0, c1);
            s8x4_to_h2(v.y, c2, c3);
            s8x4_to_h2(v.z, c4, c5);
            s8x4_to_h2(v.w, c6, c7);
            sts128(at, tc::sw128_offset(ar, 2 * aq), c0, c1, c2, c3);
            sts128(at, tc::sw128_offset(ar, 2 * aq + 1), c4, c5, c6, c7);
          }
        }
        // B: 16 quant bytes -> low sub-block chunks 2h, 2h+1 and high 4+2h, 5+2h
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) {
          const int u = ci + kConvThreads * ub;
          if (u < kUnitsB) {
            const int br = u >> 1, bh = u & 1;
            uint32_t sc_lo = 1, sc_hi = 1, mdummy;
            if (!dots_only) {
              scale_min(hdr_keep[ub][si.sb & 1], 2 * si.c, sc_lo, mdummy);
              scale_min(hdr_keep[ub][si.sb & 1], 2 * si.c + 1, sc_hi, mdummy);
            }
            const float fl = (float)sc_lo, fh = (float)sc_hi;
            const __half2 m_lo = __float2half2_rn(fl), a_lo = __float2half2_rn(-1024.0f * fl);
            const __half2 m_hi = __float2half2_rn(fh * 0.0625f), a_hi = __float2half2_rn(-64.0f * fh);
            const uint4 q = cur.v[3 + ub];
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
            uint32_t lo[4][2], hi[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) q4x8_to_h2(words[i], m_lo, a_lo, m_hi, a_hi, lo[i], hi[i]);
            sts128(bt, tc::sw128_offset(br, 2 * bh), lo[0][0], lo[0][1], lo[1][0], lo[1][1]);
            sts128(bt, tc::sw128_offset(br, 2 * bh + 1), lo[2][0], lo[2][1], lo[3][0], lo[3][1]);
            sts128(bt, tc::sw128_offset(br, 4 + 2 * bh), hi[0][0], hi[0][1], hi[1][0], hi[1][1]);
            sts128(bt, tc::sw128_offset(br, 5 + 2 * bh), hi[2][0], hi[2][1], hi[3][0], hi[3][1]);
          }
        }
      } else {
        // min-term operands of superblock si.sb + h for token / row r:
        // A = (u1,u1,u2,u2), B = (v1,v2,v1,v2) per block, u = d8*S, v = dmin*m
#pragma unroll
        for (int ub = 0; ub < 2; ++ub) {
          const int u = ci + kConvThreads * ub;
          if (u < kUnitsB) {
            const int r = u >> 1, h = u & 1;
            const uint4 dlo = cur.v[4 * ub], dhi = cur.v[4 * ub + 1];
            const uint4 slo = cur.v[4 * ub + 2], shi = cur.v[4 * ub + 3];
            const float dd[8] = {__uint_as_float(dlo.x), __uint_as_float(dlo.y), __uint_as_float(dlo.z),
                                 __uint_as_float(dlo.w), __uint_as_float(dhi.x), __uint_as_float(dhi.y),
                                 __uint_as_float(dhi.z), __uint_as_float(dhi.w)};
            const int ss[8] = {(int)slo.x, (int)slo.y, (int)slo.z, (int)slo.w,
                               (int)shi.x, (int)shi.y, (int)shi.z, (int)shi.w};
            const uint4 hh = hdr_keep[ub][h];
            const bool sb_ok = si.sb + h < nb && row0 + r < rows;
            const float dmin = sb_ok ? __half2float(__ushort_as_half((unsigned short)(hh.x >> 16))) : 0.0f;
            uint32_t av[16], bv[16];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
              float u1, u2, v1, v2;
              split_bf16(dd[b] * (float)ss[b], u1, u2);
              uint32_t scv, mv;
              scale_min(hh, b, scv, mv);
              split_bf16(dmin * (float)mv, v1, v2);
              av[2 * b] = bf16x2(u1, u1);
              av[2 * b + 1] = bf16x2(u2, u2);
              bv[2 * b] = bf16x2(v1, v2);
              bv[2 * b + 1] = bf16x2(v1, v2);
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              sts128(at, tc::sw128_offset(r, 4 * h + jj), av[4 * jj], av[4 * jj + 1], av[4 * jj + 2],
                     av[4 * jj + 3]);
              sts128(bt, tc::sw128_offset(r, 4 * h + jj), bv[4 * jj], bv[4 * jj + 1], bv[4 * jj + 2],
                     bv[4 * jj + 3]);
            }
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&sm.full[st]);
      cur = nxt;
    }
    if (!ok) fail();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 1 - kConvWarps;
    const int q = warp & 3, g = e >> 2;
    const int t = 32 * q + lane, tok = tok0 + t;
    const bool tok_ok = tok < tokens;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const int cb = 64 * g;
    float2 sb_acc[32];
    bool ok = true;
    int blk = 0;
    for (int sb = 0; sb < nb && ok; ++sb) {
      float d8v[8];
      if (tok_ok && !dots_only) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(d8 + (size_t)tok * nsub + 8 * sb));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(d8 + (size_t)tok * nsub + 8 * sb + 4));
        d8v[0] = lo.x; d8v[1] = lo.y; d8v[2] = lo.z; d8v[3] = lo.w;
        d8v[4] = hi.x; d8v[5] = hi.y; d8v[6] = hi.z; d8v[7] = hi.w;
      } else {
        for (int i = 0; i < 8; ++i) d8v[i] = 0.0f;
      }
      for (int i = 0; i < 32; ++i) sb_acc[i] = make_float2(0.0f, 0.0f);
      for (int b = 0; b < 8; ++b) {
        const int buf = blk & 1;
        if (!tc::mbar_wait(&sm.tfull[buf], (blk >> 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const float2 s2 = make_float2(d8v[b], d8v[b]);
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tc::tmem_ld32(lane_base + 128u * buf + cb + 32 * half, r);
          tc::tmem_wait_ld();
          if (dots_only) {
            if (tok_ok) {
              for (int i = 0; i < 32; ++i) {
                const int o = row0 + cb + 32 * half + i;
                if (o < rows)
                  p_out[((size_t)tok * rows + o) * nsub + blk] = (int32_t)__uint_as_float(r[i]);
              }
            }
          } else {
            for (int i = 0; i < 16; ++i)
              sb_acc[16 * half + i] = __ffma2_rn(
                  make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), s2,
                  sb_acc[16 * half + i]);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.tempty[buf]);
        ++blk;
      }
      if (!ok) break;
      // superblock done: running total += d[o] * sb_acc
      if (!tc::mbar_wait(&sm.dfull[sb & 1], (sb >> 1) & 1, abort_flag)) { ok = false; break; }
      if (!dots_only) {
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          const uint32_t taddr = lane_base + kColAcc + cb + 32 * half;
          if (sb > 0) {
            tc::tmem_ld32(taddr, r);
            tc::tmem_wait_ld();
          } else {
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          const float4* dp = reinterpret_cast<const float4*>(&sm.dsm[sb & 1][cb + 32 * half]);
          for (int i = 0; i < 8; ++i) {
            const float4 dv = dp[i];
            const float2 a0 = __ffma2_rn(sb_acc[16 * half + 2 * i], make_float2(dv.x, dv.y),
                                         make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])));
            const float2 a1 = __ffma2_rn(sb_acc[16 * half + 2 * i + 1], make_float2(dv.z, dv.w),
                                         make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
            r[4 * i] = __float_as_uint(a0.x);
            r[4 * i + 1] = __float_as_uint(a0.y);
            r[4 * i + 2] = __float_as_uint(a1.x);
            r[4 * i + 3] = __float_as_uint(a1.y);
          }
          tc::tmem_st32(taddr, r);
          tc::tmem_wait_st();
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.dempty[sb & 1]);
    }
    if (ok && !dots_only) {
      if (!tc::mbar_wait(&sm.mfull, 0, abort_flag)) ok = false;
      if (ok) {
        tc::fence_after_sync();
        for (int half = 0; half < 2; ++half) {
          uint32_t ra[32], rm[32];
          tc::tmem_ld32(lane_base + kColAcc + cb + 32 * half, ra);
          tc::tmem_ld32(lane_base + kColMin + cb + 32 * half, rm);
          tc::tmem_wait_ld();
          if (tok_ok) {
            const int o0 = row0 + cb + 32 * half;
            float* yrow = y + (size_t)tok * rows + o0;
            if (o0 + 32 <= rows && (rows & 3) == 0) {
              for (int i = 0; i < 8; ++i) {
                float4 v;
                v.x = __uint_as_float(ra[4 * i]) - __uint_as_float(rm[4 * i]);
                v.y = __uint_as_float(ra[4 * i + 1]) - __uint_as_float(rm[4 * i + 1]);
                v.z = __uint_as_float(ra[4 * i + 2]) - __uint_as_float(rm[4 * i + 2]);
                v.w = __uint_as_float(ra[4 * i + 3]) - __uint_as_float(rm[4 * i + 3]);
                reinterpret_cast<float4*>(yrow)[i] = v;
              }
            } else {
              for (int i = 0; i < 32; ++i)
                if (o0 + i < rows) yrow[i] = __uint_as_float(ra[i]) - __uint_as_float(rm[i]);
            }
          }
        }
      }
    }
    if (!ok) fail();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool gemm_tc_supported(int64_t tokens) { return tokens >= 16; }

cudaError_t launch_gemm_block144(const uint8_t* w, int64_t rows, int64_t cols,
                                 const int8_t* q8, const float* d8,
                                 const int32_t* sum, int64_t tokens, float* y,
                                 int32_t* p_out, int* err, cudaStream_t s) {
  if (rows == 0 || tokens == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = sizeof(Smem) + 1024;
  static int s_set[64];
  if (!s_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    s_set[dev & 63] = 1;
  }
  dim3 grid((unsigned)((rows + kBN - 1) / kBN), (unsigned)((tokens + kBM - 1) / kBM));
  gemm_tc_kernel<<<grid, kThreads, smem, s>>>(w, (int)rows, (int)(cols / kQK), q8, d8, sum,
                                              (int)tokens, y, p_out, err);
  return cudaGetLastError();
}

}  // namespace q4k
