// q4k_gemm_h16 on the sm_103a tensor cores: the prefill MMQ GEMM over q8_1
// activations whose quants arrive as exact binary16 integers
// (q8_quantize_h16), the operand form the tensor core reads (genie-ai-runtime
// §3, "The tensor-core kernel (Path E)" is the prior art; this is the
// integer MMQ form of it).
//
//   y[t][o] = sum_b d*sc[o,b] * d8[t,b] * P[t,o,b] - dmin*m[o,b] * d8[t,b] * S[t,b]
//   P[t,o,b] = sum_{i<32} q[o][32b+i] * q8[t][32b+i]
//
// The integer dots run on tcgen05.mma kind::f16 with operands that are exact
// small integers: A = q8 (|q8| <= 127) and B = sc*q (<= 63*15 = 945), both
// exact in fp16, so every product and partial sum of one 32-wide block
// (|sum| < 2^22) is an integer fp32 holds exactly and a block's TMEM
// accumulator equals sc*P whatever order the tensor core adds in.
//
// Tile: 128 tokens (TMEM lanes) x 128 weight rows (TMEM columns); K walks
// 64 weights (one 128-byte swizzle atom of fp16) per pipeline stage.  The A
// tile of a stage is one tensor copy straight into the 128-byte-swizzled
// K-major layout the MMA reads: nothing converts the activations.  Warp
// roles in one CTA of 14 warps:
//   warp 0      lane 0 issues every tensor copy: A stages, one raw
//               128-row x 144-byte superblock tile per superblock, d8 and
//               block-sum tiles
//   warp 1      allocates TMEM; lane 0 issues every tcgen05.mma
//   warps 2-5   converters, thread i = weight row i and token i of the tile:
//               widen row i's quants to sc*q fp16 in the swizzled layout,
//               hand each superblock's d (per row) and d8 (per token,
//               block-major) to the epilogue, and build the min-term operands
//   warps 6-13  epilogue: per block, read the block's accumulator from TMEM
//               and add it, times the token's scale d8, into a per-superblock
//               sum in registers; per superblock, add d * sum into a running
//               fp32 total kept in TMEM
// TMEM columns: [0,128) and [128,256) double-buffered block accumulators,
// [256,384) the min-term accumulator, [384,512) the running total.
//
// The min term sum_b (dmin*m[o,b]) * (d8*S[t,b]) is a depth-(K/32) product;
// it runs on the tensor cores too (bf16, both factors split into two bf16
// parts, 4 products per block, ~2^-16 relative error), one extra MMA group
// after every two superblocks, from its own operand buffers.
//
// Every mbarrier wait is bounded (tc::kTimeoutCycles); a wait that gives up
// sets the library's device error word, raises a CTA-wide abort flag and the
// CTA unwinds, drains its MMAs and tensor copies and frees its TMEM.
#include "mmq_cvt.cuh"
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kBM = 128;                 // tokens per tile
constexpr int kBN = 128;                 // weight rows per tile
constexpr int kAStages = 4;              // fp16 q8 operand stages (tensor copies)
constexpr int kBStages = 3;              // fp16 sc*q operand stages (converted)
constexpr int kBRaw = 2;                 // raw superblock tiles in flight
constexpr int kTileBytes = 128 * 128;    // 128 rows x 64 k x fp16
constexpr int kBRawBytes = kBN * kBlockBytes;
constexpr int kD8RawBytes = kBM * 32;    // 128 tokens x 8 fp32: d8 of one superblock
constexpr int kSRawBytes = kBM * 64;     // 128 tokens x 16 int32: sums of a superblock pair
constexpr int kConvWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 32 * (2 + kConvWarps + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColMin = 256;
constexpr uint32_t kColAcc = 384;
static_assert(kConvThreads == kBN && kConvThreads == kBM, "one converter thread per row and per token");

struct __align__(1024) Smem {
  uint8_t a[kAStages][kTileBytes];         // fp16 q8 operand, 128B-swizzled (tensor copies)
  uint8_t b[kBStages][kTileBytes];         // fp16 sc*q operand, 128B-swizzled
  uint8_t amin[kTileBytes];                // bf16 min-term operands
  uint8_t bmin[kTileBytes];
  uint8_t braw[kBRaw][kBRawBytes];         // superblocks as copied
  float d8raw[2][kBM][8];                  // d8 of a superblock, as copied
  float d8t[2][8][kBM];                    // the same, block-major, by superblock parity
  int32_t sraw[kBM][16];                   // block sums of a superblock pair
  float dsm[2][kBN];                       // d of each row, by superblock parity
  uint64_t afull[kAStages], aempty[kAStages];
  uint64_t bfull[kBStages], bempty[kBStages];
  uint64_t rfull[kBRaw], rempty[kBRaw];
  uint64_t d8full[2], d8empty[2], sfull, sempty;
  uint64_t minfull, minempty;
  uint64_t tfull[2], tempty[2];
  uint64_t dfull[2], dempty[2];
  uint64_t mfull, drain;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per CTA, plus the 1024-byte alignment pad
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// f = hi + lo with hi = bf16(f) and lo = bf16(f - hi)
__device__ __forceinline__ void split_bf16(float f, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(f));
  lo = __bfloat162float(__float2bfloat16_rn(f - hi));
}

// acc += (a, b) * s2 as one fp32x2 FMA
__device__ __forceinline__ void ffma2_acc(uint64_t& acc, uint32_t a, uint32_t b, uint64_t s2) {
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tfma.rn.f32x2 %0, t, %3, %0;\n\t}"
      : "+l"(acc) : "r"(a), "r"(b), "l"(s2));
}

// (r0, r1) = acc * (d0, d1) + (r0, r1)
__device__ __forceinline__ void ffma2_into(uint32_t& r0, uint32_t& r1, uint64_t acc, float d0, float d1) {
  asm("{\n\t.reg .b64 t, dd;\n\tmov.b64 t, {%0, %1};\n\tmov.b64 dd, {%2, %3};\n\t"
      "fma.rn.f32x2 t, %4, dd, t;\n\tmov.b64 {%0, %1}, t;\n\t}"
      : "+r"(r0), "+r"(r1) : "f"(d0), "f"(d1), "l"(acc));
}

__device__ __forceinline__ uint64_t pack2(float a, float b) {
  return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}

using namespace cvt;

struct GemmParams {
  CUtensorMap map_a;    // fp16 q8 {K, tokens}, box {64, 128}, 128-byte swizzle
  CUtensorMap map_b;    // superblocks {144, rows, nb}, box {144, 128, 1}
  CUtensorMap map_d8;   // d8 bytes {K/8, tokens, 1}, box {32, 128, 1}
  CUtensorMap map_s;    // block sums, bytes {K/8, tokens, 1}, box {64, 128, 1}
  float* y;
  int32_t* p_out;       // non-null: store the per-block integer dots instead
  int* err;
  int rows, nb, tokens;
};

__global__ void __launch_bounds__(kThreads, 1) gemm_h16_kernel(const __grid_constant__ GemmParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &sm.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kBN, tok0 = blockIdx.y * kBM;
  const int nb = P.nb, rows = P.rows, tokens = P.tokens;
  const int nsub = 8 * nb;
  const bool dots_only = P.p_out != nullptr;
  const bool with_min = !dots_only;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAStages; ++i) {
      tc::mbar_init(&sm.afull[i], 1);
      tc::mbar_init(&sm.aempty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      tc::mbar_init(&sm.bfull[i], kConvThreads);
      tc::mbar_init(&sm.bempty[i], 1);
    }
    for (int i = 0; i < kBRaw; ++i) {
      tc::mbar_init(&sm.rfull[i], 1);
      tc::mbar_init(&sm.rempty[i], kConvThreads);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.d8full[i], 1);
      tc::mbar_init(&sm.d8empty[i], kConvThreads);
      tc::mbar_init(&sm.tfull[i], 1);
      tc::mbar_init(&sm.tempty[i], kEpiWarps);
      tc::mbar_init(&sm.dfull[i], kConvThreads);
      tc::mbar_init(&sm.dempty[i], kEpiWarps);
    }
    tc::mbar_init(&sm.sfull, 1);
    tc::mbar_init(&sm.sempty, kConvThreads);
    tc::mbar_init(&sm.minfull, kConvThreads);
    tc::mbar_init(&sm.minempty, 1);
    tc::mbar_init(&sm.mfull, 1);
    tc::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  auto fail = [&]() {
    if (!*abort_flag) atomicOr(P.err, 1);
    *abort_flag = 1;
  };
  // the superblock after which a min-term group runs (each odd one, and the last)
  auto min_after = [&](int sb) { return with_min && ((sb & 1) || sb == nb - 1); };

  if (warp == 0) {
    // --------------------------------------------------------- tensor copies
    if (lane == 0) {
      bool ok = true;
      int na = 0, nr = 0, nd = 0, ns = 0;   // copies issued
      for (int sb = 0; sb < nb && ok; ++sb) {
        {
          const int slot = sb % kBRaw;
          if (!tc::mbar_wait(&sm.rempty[slot], ((sb / kBRaw) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.rfull[slot], kBRawBytes);
          tc::tma_load_3d(sm.braw[slot], &P.map_b, 0, row0, sb, &sm.rfull[slot]);
          ++nr;
        }
        if (with_min) {
          const int slot = sb & 1;
          if (!tc::mbar_wait(&sm.d8empty[slot], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.d8full[slot], kD8RawBytes);
          tc::tma_load_3d(sm.d8raw[slot], &P.map_d8, 32 * sb, tok0, 0, &sm.d8full[slot]);
          ++nd;
          if ((sb & 1) == 0) {
            if (!tc::mbar_wait(&sm.sempty, ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            tc::mbar_arrive_expect_tx(&sm.sfull, kSRawBytes);
            tc::tma_load_3d(sm.sraw, &P.map_s, 64 * (sb >> 1), tok0, 0, &sm.sfull);
            ++ns;
          }
        }
        for (int c = 0; c < 4; ++c) {
          const int j = 4 * sb + c, slot = j % kAStages;
          if (!tc::mbar_wait(&sm.aempty[slot], ((j / kAStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.afull[slot], kTileBytes);
          tc::tma_load_2d(sm.a[slot], &P.map_a, 64 * j, tok0, &sm.afull[slot]);
          ++na;
        }
      }
      if (!ok) fail();
      // every copy issued lands before the CTA exits (after an abort some
      // were never consumed)
      bool drained = true;
      for (int j = na - 1; j >= 0 && j >= na - kAStages; --j)
        drained &= tc::mbar_wait_sleep(&sm.afull[j % kAStages], (j / kAStages) & 1);
      for (int sb = nr - 1; sb >= 0 && sb >= nr - kBRaw; --sb)
        drained &= tc::mbar_wait_sleep(&sm.rfull[sb % kBRaw], (sb / kBRaw) & 1);
      for (int sb = nd - 1; sb >= 0 && sb >= nd - 2; --sb)
        drained &= tc::mbar_wait_sleep(&sm.d8full[sb & 1], (sb >> 1) & 1);
      if (ns > 0) drained &= tc::mbar_wait_sleep(&sm.sfull, (ns - 1) & 1);
      if (!drained) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idf = tc::idesc_f16(kBM, kBN, false);
      const uint32_t idb = tc::idesc_f16(kBM, kBN, true);
      bool ok = true;
      int blk = 0;
      for (int sb = 0; sb < nb && ok; ++sb) {
        for (int c = 0; c < 4 && ok; ++c) {
          const int j = 4 * sb + c, sa = j % kAStages, sbs = j % kBStages;
          if (!tc::mbar_wait(&sm.afull[sa], (j / kAStages) & 1, abort_flag) ||
              !tc::mbar_wait(&sm.bfull[sbs], (j / kBStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_base = tc::smem_u32(sm.a[sa]), b_base = tc::smem_u32(sm.b[sbs]);
          for (int h = 0; h < 2; ++h) {
            const int buf = blk & 1;
            if (!tc::mbar_wait(&sm.tempty[buf], ((blk >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t koff = (uint32_t)(2 * h + kk) * 32u;
              tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_base + koff), tc::desc_sw128(b_base + koff), idf,
                             (uint32_t)kk);
            }
            tc::mma_commit(&sm.tfull[buf]);
            ++blk;
          }
          if (!ok) break;
          tc::mma_commit(&sm.aempty[sa]);
          tc::mma_commit(&sm.bempty[sbs]);
        }
        if (ok && min_after(sb)) {
          const int p = sb >> 1;
          if (!tc::mbar_wait(&sm.minfull, p & 1, abort_flag)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a_base = tc::smem_u32(sm.amin), b_base = tc::smem_u32(sm.bmin);
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f16_ss(tmem + kColMin, tc::desc_sw128(a_base + 32u * kk), tc::desc_sw128(b_base + 32u * kk),
                           idb, (p > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&sm.minempty);
        }
      }
      if (!ok) fail();
      tc::mma_commit(&sm.mfull);
      // every MMA issued above completes before TMEM is freed
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait_sleep(&sm.drain, 0)) fail();
    }
  } else if (warp < 2 + kConvWarps) {
    // ------------------------------------------------------------ converters
    const int ci = threadIdx.x - 64;             // weight row ci and token ci of the tile
    uint32_t m03_0 = 0, m47_0 = 0, m03_1 = 0, m47_1 = 0, dmin_0 = 0, dmin_1 = 0;
    bool ok = true;
    for (int sb = 0; sb < nb && ok; ++sb) {
      const int rslot = sb % kBRaw;
      if (!tc::mbar_wait(&sm.rfull[rslot], (sb / kBRaw) & 1, abort_flag)) { ok = false; break; }
      const uint8_t* raw_row = sm.braw[rslot] + ci * kBlockBytes;
      const uint4 hd = *reinterpret_cast<const uint4*>(raw_row);
      uint32_t sc03, sc47, m03, m47;
      header_sc_m(hd, sc03, sc47, m03, m47);
      if (dots_only) sc03 = sc47 = 0x01010101u;
      if (sb & 1) { m03_1 = m03; m47_1 = m47; dmin_1 = hd.x >> 16; }
      else { m03_0 = m03; m47_0 = m47; dmin_0 = hd.x >> 16; }
      if (with_min) {
        // hand the epilogue this superblock's d (per row) and d8 (per token,
        // block-major) once it is done with superblock sb - 2
        const int par = sb & 1;
        if (!tc::mbar_wait(&sm.d8full[par], (sb >> 1) & 1, abort_flag)) { ok = false; break; }
        const float4 dlo = *reinterpret_cast<const float4*>(&sm.d8raw[par][ci][0]);
        const float4 dhi = *reinterpret_cast<const float4*>(&sm.d8raw[par][ci][4]);
        tc::mbar_arrive(&sm.d8empty[par]);
        if (!tc::mbar_wait(&sm.dempty[par], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        sm.dsm[par][ci] = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
        sm.d8t[par][0][ci] = dlo.x; sm.d8t[par][1][ci] = dlo.y;
        sm.d8t[par][2][ci] = dlo.z; sm.d8t[par][3][ci] = dlo.w;
        sm.d8t[par][4][ci] = dhi.x; sm.d8t[par][5][ci] = dhi.y;
        sm.d8t[par][6][ci] = dhi.z; sm.d8t[par][7][ci] = dhi.w;
        tc::mbar_arrive(&sm.dfull[par]);
      }
      for (int c = 0; c < 4; ++c) {
        const int j = 4 * sb + c, slot = j % kBStages;
        const uint4 q0 = *reinterpret_cast<const uint4*>(raw_row + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(raw_row + 32 + 32 * c);
        if (c == 3) tc::mbar_arrive(&sm.rempty[rslot]);
        if (!tc::mbar_wait(&sm.bempty[slot], ((j / kBStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
        uint8_t* bt = sm.b[slot];
        // sub-blocks 2c (low nibbles, k 0..31 of the stage) and 2c+1 (high, k 32..63)
        const uint32_t scw = c < 2 ? sc03 : sc47;
        const uint32_t bsel = 2u * (uint32_t)(c & 1);
        const uint32_t slo = byte_h2(scw, bsel), shi = byte_h2(scw, bsel + 1);
        const uint32_t mlo = slo, alo = mul_h2(slo, 0xE400E400u);   // -1024
        const uint32_t mhi = mul_h2(shi, 0x2C002C00u);              // 1/16
        const uint32_t ahi = mul_h2(shi, 0xD400D400u);              // -64
        uint32_t l0, l1, l2, l3, l4, l5, l6, l7, h0, h1, h2, h3, h4, h5, h6, h7;
        cvt_q4x8(q0.x, mlo, alo, mhi, ahi, l0, l1, h0, h1);
        cvt_q4x8(q0.y, mlo, alo, mhi, ahi, l2, l3, h2, h3);
        cvt_q4x8(q0.z, mlo, alo, mhi, ahi, l4, l5, h4, h5);
        cvt_q4x8(q0.w, mlo, alo, mhi, ahi, l6, l7, h6, h7);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 0)) = make_uint4(l0, l1, l2, l3);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 1)) = make_uint4(l4, l5, l6, l7);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 4)) = make_uint4(h0, h1, h2, h3);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 5)) = make_uint4(h4, h5, h6, h7);
        cvt_q4x8(q1.x, mlo, alo, mhi, ahi, l0, l1, h0, h1);
        cvt_q4x8(q1.y, mlo, alo, mhi, ahi, l2, l3, h2, h3);
        cvt_q4x8(q1.z, mlo, alo, mhi, ahi, l4, l5, h4, h5);
        cvt_q4x8(q1.w, mlo, alo, mhi, ahi, l6, l7, h6, h7);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 2)) = make_uint4(l0, l1, l2, l3);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 3)) = make_uint4(l4, l5, l6, l7);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 6)) = make_uint4(h0, h1, h2, h3);
        *reinterpret_cast<uint4*>(bt + tc::sw128_offset(ci, 7)) = make_uint4(h4, h5, h6, h7);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&sm.bfull[slot]);
      }
      if (!ok) break;
      if (min_after(sb)) {
        // min-term operands of superblocks 2p, 2p+1: per block, A = (u1,u1,u2,u2)
        // with u = d8*S split into bf16 hi + lo (token ci), B = (v1,v2,v1,v2)
        // with v = dmin*m split the same way (row ci); the four products sum to u*v
        const int p = sb >> 1;
        if (!tc::mbar_wait(&sm.sfull, p & 1, abort_flag)) { ok = false; break; }
        uint32_t av[32];
        const int32_t* sp = sm.sraw[ci];
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          // a missing second superblock contributes 0
          float u1 = 0.0f, u2 = 0.0f;
          if (b < 8 || 2 * p + 1 < nb) split_bf16(sm.d8t[b >> 3][b & 7][ci] * (float)sp[b], u1, u2);
          av[2 * b] = bf16x2(u1, u1);
          av[2 * b + 1] = bf16x2(u2, u2);
        }
        tc::mbar_arrive(&sm.sempty);
        if (!tc::mbar_wait(&sm.minempty, (p & 1) ^ 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          *reinterpret_cast<uint4*>(sm.amin + tc::sw128_offset(ci, jj)) =
              make_uint4(av[4 * jj], av[4 * jj + 1], av[4 * jj + 2], av[4 * jj + 3]);
        const bool row_ok = row0 + ci < rows;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const bool sb_ok = row_ok && 2 * p + h < nb;
          const float dmin = sb_ok ? __half2float(__ushort_as_half((unsigned short)(h ? dmin_1 : dmin_0))) : 0.0f;
          const uint32_t mA = h ? m03_1 : m03_0, mB = h ? m47_1 : m47_0;
          uint32_t bv[16];
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const uint32_t mv = ((b < 4 ? mA : mB) >> (8 * (b & 3))) & 0xFFu;
            float v1, v2;
            split_bf16(dmin * (float)mv, v1, v2);
            bv[2 * b] = bf16x2(v1, v2);
            bv[2 * b + 1] = bv[2 * b];
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<uint4*>(sm.bmin + tc::sw128_offset(ci, 4 * h + jj)) =
                make_uint4(bv[4 * jj], bv[4 * jj + 1], bv[4 * jj + 2], bv[4 * jj + 3]);
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&sm.minfull);
      }
    }
    if (!ok) fail();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2 - kConvWarps;
    const int q = warp & 3, g = e >> 2;          // TMEM lane quarter (warp % 4), column half
    const int t = 32 * q + lane, tok = tok0 + t;
    const bool tok_ok = tok < tokens;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const int cb = 64 * g;
    bool ok = true;
    if (dots_only) {
      // test export: store each block's integer dots
      for (int blk = 0; blk < nsub && ok; ++blk) {
        const int buf = blk & 1;
        if (!tc::mbar_wait(&sm.tfull[buf], (blk >> 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tc::tmem_ld32(lane_base + 128u * buf + cb + 32 * half, r);
          tc::tmem_wait_ld();
          if (tok_ok) {
            for (int i = 0; i < 32; ++i) {
              const int o = row0 + cb + 32 * half + i;
              if (o < rows) P.p_out[((size_t)tok * rows + o) * nsub + blk] = (int32_t)__uint_as_float(r[i]);
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.tempty[buf]);
      }
    }
    uint64_t acc[32];   // per-superblock sum, pairs of rows
    int blk = 0;
    for (int sb = 0; sb < nb && ok && !dots_only; ++sb) {
      // d8 (block-major) and d of this superblock, from the converters
      if (!tc::mbar_wait(&sm.dfull[sb & 1], (sb >> 1) & 1, abort_flag)) { ok = false; break; }
      const float* d8c = &sm.d8t[sb & 1][0][t];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0ull;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int buf = blk & 1;
        if (!tc::mbar_wait(&sm.tfull[buf], (blk >> 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const float d8b = d8c[b * kBM];
        const uint64_t s2 = pack2(d8b, d8b);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tc::tmem_ld32(lane_base + 128u * buf + cb + 32 * half, r);
          tc::tmem_wait_ld();
          if (half == 1) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm.tempty[buf]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) ffma2_acc(acc[16 * half + i], r[2 * i], r[2 * i + 1], s2);
        }
        ++blk;
      }
      if (!ok) break;
      // superblock done: running total += d[o] * acc
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t r[16];
        const uint32_t taddr = lane_base + kColAcc + cb + 16 * qq;
        if (sb > 0) {
          tc::tmem_ld16(taddr, r);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = 0u;
        }
        const float4* dp = reinterpret_cast<const float4*>(&sm.dsm[sb & 1][cb + 16 * qq]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 dv = dp[i];
          ffma2_into(r[4 * i], r[4 * i + 1], acc[8 * qq + 2 * i], dv.x, dv.y);
          ffma2_into(r[4 * i + 2], r[4 * i + 3], acc[8 * qq + 2 * i + 1], dv.z, dv.w);
        }
        tc::tmem_st16(taddr, r);
      }
      tc::tmem_wait_st();
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
            float* yrow = P.y + (size_t)tok * rows + o0;
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
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm_h16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* q16, const float* d8,
                            const int32_t* sum, int64_t tokens, float* y, int32_t* p_out, int* err,
                            cudaStream_t s) {
  if (rows == 0 || tokens == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = sizeof(Smem) + 1024;
  static int s_set[64];
  if (!s_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_h16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    s_set[dev & 63] = 1;
  }
  const int64_t nb = cols / kQK;
  GemmParams P{};
  if (!encode_tmap_2d(&P.map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q16, (uint64_t)cols, (uint64_t)tokens,
                      (uint64_t)cols * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)nb * kBlockBytes, (uint64_t)kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, kBN, 1};
    if (!encode_tmap_u8_3d(&P.map_b, w, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if (!p_out) {
    const uint64_t rb = (uint64_t)(cols / kSub) * 4;   // bytes of one token's d8 (or sums)
    const uint64_t dims[3] = {rb, (uint64_t)tokens, 1};
    const uint64_t strides[2] = {rb, rb * (uint64_t)tokens};
    const uint32_t box_d8[3] = {kD8RawBytes / kBM, kBM, 1};   // one superblock's 8 blocks
    const uint32_t box_s[3] = {kSRawBytes / kBM, kBM, 1};     // a superblock pair's 16 blocks
    if (!encode_tmap_u8_3d(&P.map_d8, d8, dims, strides, box_d8)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8_3d(&P.map_s, sum, dims, strides, box_s)) return cudaErrorInvalidValue;
  }
  P.y = y;
  P.p_out = p_out;
  P.err = err;
  P.rows = (int)rows;
  P.nb = (int)nb;
  P.tokens = (int)tokens;
  dim3 grid((unsigned)((rows + kBN - 1) / kBN), (unsigned)((tokens + kBM - 1) / kBM));
  gemm_h16_kernel<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace q4k
