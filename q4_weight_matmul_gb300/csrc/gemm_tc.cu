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
//   warp 0      allocates TMEM; lane 0 issues the tensor copies (raw q8 tile
//               of each stage, one 128-row x 144-byte superblock tile per
//               superblock, d8 and block-sum tiles) and every tcgen05.mma
//   warps 1-7   converters: read the raw tiles from shared memory, widen them
//               to fp16 (B pre-multiplied by sc) and store them in the
//               128-byte-swizzled K-major layout the MMA reads; hand each
//               superblock's d (per row) and d8 (per token, block-major) to
//               the epilogue
//   warps 8-15  epilogue: per block, read the block's accumulator from TMEM
//               and add it, times the token's scale d8, into a per-superblock
//               sum in registers; per superblock, add d * sum into a running
//               fp32 total kept in TMEM
// TMEM columns: [0,128) and [128,256) double-buffered block accumulators,
// [256,384) the min-term accumulator, [384,512) the running total.
//
// The min term sum_b (dmin*m[o,b]) * (d8*S[t,b]) is a depth-(K/32) product;
// it runs on the tensor cores too (bf16, both factors split into two bf16
// parts, 4 products per block, ~2^-16 relative error), one extra stage after
// every two superblocks, into its own accumulator.
//
// Every mbarrier wait is bounded (tc::kTimeoutCycles); a wait that gives up
// sets the library's device error word, raises a CTA-wide abort flag and the
// CTA unwinds, drains its MMAs and tensor copies and frees its TMEM.
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kBM = 128;                 // tokens per tile
constexpr int kBN = 128;                 // weight rows per tile
constexpr int kStages = 3;               // fp16 operand stages
constexpr int kARaw = 6;                 // raw q8 tiles in flight
constexpr int kBRaw = 3;                 // raw superblock tiles in flight
constexpr int kTileBytes = 128 * 128;    // 128 rows x 64 k x fp16
constexpr int kARawBytes = kBM * 64;     // 128 tokens x 64 int8
constexpr int kBRawBytes = kBN * kBlockBytes;
constexpr int kD8RawBytes = kBM * 32;    // 128 tokens x 8 fp32: d8 of one superblock
constexpr int kSRawBytes = kBM * 64;     // 128 tokens x 16 int32: sums of a superblock pair
constexpr int kConvWarps = 7;
constexpr int kEpiWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kXThreads = 96;            // converters that only widen q8
constexpr int kZThreads = 128;           // converters that own a weight row
constexpr int kTokThreads = 128;         // converters that own a token: X and the first Z warp
constexpr int kThreads = 32 * (1 + kConvWarps + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColMin = 256;
constexpr uint32_t kColAcc = 384;
static_assert(kXThreads + kZThreads == kConvThreads, "converter split");
static_assert(kXThreads * 5 + 32 == 4 * kBM, "q8 units per stage");

struct __align__(1024) Smem {
  uint8_t a[kStages][kTileBytes];          // fp16 q8 operand, 128B-swizzled
  uint8_t b[kStages][kTileBytes];          // fp16 sc*q operand, 128B-swizzled
  uint8_t araw[kARaw][kARawBytes];         // q8 tiles as copied
  uint8_t braw[kBRaw][kBRawBytes];         // superblocks as copied
  float d8raw[2][kBM][8];                  // d8 of a superblock, as copied
  float d8t[2][8][kBM];                    // the same, block-major, by superblock parity
  int32_t sraw[kBM][16];                   // block sums of a superblock pair
  float dsm[2][kBN];                       // d of each row, by superblock parity
  uint64_t full[kStages], empty[kStages];
  uint64_t afull[kARaw], aempty[kARaw];
  uint64_t bfull[kBRaw], bempty[kBRaw];
  uint64_t d8full[2], d8empty[2], sfull, sempty;
  uint64_t tfull[2], tempty[2];
  uint64_t dfull[2], dempty[2];
  uint64_t mfull, drain;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per CTA, plus the 1024-byte alignment pad
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

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

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// f = hi + lo with hi = bf16(f) and lo = bf16(f - hi)
__device__ __forceinline__ void split_bf16(float f, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(f));
  lo = __bfloat162float(__float2bfloat16_rn(f - hi));
}

// 16 int8 (k0..k15) -> two 16-byte fp16 chunks, each pair ordered (k,k+2),
// (k+1,k+3): bias each byte by 128, place it under the fp16 exponent of
// 1024 and subtract 1152.
__device__ __forceinline__ void cvt_s8x16(const uint4& v, uint4& c0, uint4& c1) {
  asm("{\n\t.reg .b32 u0,u1,u2,u3,mg,of;\n\t"
      "mov.b32 mg, 0x64646464;\n\tmov.b32 of, 0x64806480;\n\t"
      "xor.b32 u0, %8, 0x80808080;\n\txor.b32 u1, %9, 0x80808080;\n\t"
      "xor.b32 u2, %10, 0x80808080;\n\txor.b32 u3, %11, 0x80808080;\n\t"
      "prmt.b32 %0, u0, mg, 0x4240;\n\tprmt.b32 %1, u0, mg, 0x4341;\n\t"
      "prmt.b32 %2, u1, mg, 0x4240;\n\tprmt.b32 %3, u1, mg, 0x4341;\n\t"
      "prmt.b32 %4, u2, mg, 0x4240;\n\tprmt.b32 %5, u2, mg, 0x4341;\n\t"
      "prmt.b32 %6, u3, mg, 0x4240;\n\tprmt.b32 %7, u3, mg, 0x4341;\n\t"
      "sub.rn.f16x2 %0, %0, of;\n\tsub.rn.f16x2 %1, %1, of;\n\t"
      "sub.rn.f16x2 %2, %2, of;\n\tsub.rn.f16x2 %3, %3, of;\n\t"
      "sub.rn.f16x2 %4, %4, of;\n\tsub.rn.f16x2 %5, %5, of;\n\t"
      "sub.rn.f16x2 %6, %6, of;\n\tsub.rn.f16x2 %7, %7, of;\n\t}"
      : "=r"(c0.x), "=r"(c0.y), "=r"(c0.z), "=r"(c0.w), "=r"(c1.x), "=r"(c1.y), "=r"(c1.z), "=r"(c1.w)
      : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// One word of quant bytes -> sc*q fp16 pairs: low nibbles (weights l..l+3
// of the low sub-block) as (l,l+2),(l+1,l+3) in lo0/lo1, high nibbles the
// same in hi0/hi1.  Low nibbles sit under the exponent of 1024 as 1024+q,
// high nibbles as 1024+16q; one exact FMA removes the bias and applies sc.
__device__ __forceinline__ void cvt_q4x8(uint32_t w, uint32_t mlo, uint32_t alo, uint32_t mhi,
                                         uint32_t ahi, uint32_t& lo0, uint32_t& lo1, uint32_t& hi0,
                                         uint32_t& hi1) {
  asm("{\n\t.reg .b32 w8;\n\tshr.b32 w8, %4, 8;\n\t"
      "lop3.b32 %0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %1, w8, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %2, %4, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %3, w8, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "fma.rn.f16x2 %0, %0, %5, %6;\n\tfma.rn.f16x2 %1, %1, %5, %6;\n\t"
      "fma.rn.f16x2 %2, %2, %7, %8;\n\tfma.rn.f16x2 %3, %3, %7, %8;\n\t}"
      : "=r"(lo0), "=r"(lo1), "=r"(hi0), "=r"(hi1)
      : "r"(w), "r"(mlo), "r"(alo), "r"(mhi), "r"(ahi));
}

// fp16x2 (v, v) of byte `bi` of w (an integer 0..255, exact): the byte
// under the exponent of 1024, minus 1024
__device__ __forceinline__ uint32_t byte_h2(uint32_t w, uint32_t bi) {
  const uint32_t sel = bi | 0x40u | (bi << 8) | 0x4000u;   // bytes [bi, 0, bi, 0]
  uint32_t r;
  asm("{\n\t.reg .b32 t, z, k;\n\tmov.b32 z, 0;\n\tmov.b32 k, 0x64006400;\n\t"
      "prmt.b32 t, %1, z, %2;\n\tor.b32 t, t, k;\n\tsub.rn.f16x2 %0, t, k;\n\t}"
      : "=r"(r) : "r"(w), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t mul_h2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
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

// packed 6-bit scales / mins of sub-blocks 0..3 and 4..7 of a header
__device__ __forceinline__ void header_sc_m(const uint4& h, uint32_t& sc03, uint32_t& sc47, uint32_t& m03,
                                            uint32_t& m47) {
  sc03 = h.y & 0x3F3F3F3Fu;
  m03 = h.z & 0x3F3F3F3Fu;
  sc47 = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
  m47 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
}

struct GemmParams {
  CUtensorMap map_a;    // q8 bytes {K, tokens, 1}, box {64, 128, 1}
  CUtensorMap map_b;    // superblocks {144, rows, nb}, box {144, 128, 1}
  CUtensorMap map_d8;   // d8 bytes {K/8, tokens, 1}, box {32, 128, 1}
  CUtensorMap map_s;    // block sums, bytes {K/8, tokens, 1}, box {64, 128, 1}
  float* y;
  int32_t* p_out;       // non-null: store the per-block integer dots instead
  int* err;
  int rows, nb, tokens;
};

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps every access below in the shared state space
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &sm.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kBN, tok0 = blockIdx.y * kBM;
  const int nb = P.nb, rows = P.rows, tokens = P.tokens;
  const int nsub = 8 * nb;
  const bool dots_only = P.p_out != nullptr;
  const bool with_min = !dots_only;
  const int n_main = 4 * nb;
  const int n_stages = with_min ? n_main + (nb + 1) / 2 : n_main;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&sm.full[i], kConvThreads);
      tc::mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < kARaw; ++i) {
      tc::mbar_init(&sm.afull[i], 1);
      tc::mbar_init(&sm.aempty[i], kConvThreads);
    }
    for (int i = 0; i < kBRaw; ++i) {
      tc::mbar_init(&sm.bfull[i], 1);
      tc::mbar_init(&sm.bempty[i], kZThreads);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.d8full[i], 1);
      tc::mbar_init(&sm.d8empty[i], kTokThreads);
      tc::mbar_init(&sm.tfull[i], 1);
      tc::mbar_init(&sm.tempty[i], kEpiWarps);
      tc::mbar_init(&sm.dfull[i], kConvThreads);
      tc::mbar_init(&sm.dempty[i], kEpiWarps);
    }
    tc::mbar_init(&sm.sfull, 1);
    tc::mbar_init(&sm.sempty, kConvThreads);
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
    if (!*abort_flag) atomicOr(P.err, 1);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------- MMA issuer + TMA producer
    if (lane == 0) {
      const uint32_t idf = tc::idesc_f16(kBM, kBN, false);
      const uint32_t idb = tc::idesc_f16(kBM, kBN, true);
      bool ok = true;
      int a_next = 0, b_next = 0, d_next = 0, s_next = 0;   // tensor copies issued so far
      // raw q8 tile of main stage a_next, raw superblock b_next, d8 tile of
      // superblock d_next, block-sum tile of superblock pair s_next
      auto issue_a = [&]() {
        const int j = a_next, slot = j % kARaw;
        if (!tc::mbar_wait(&sm.aempty[slot], ((j / kARaw) & 1) ^ 1, abort_flag)) return false;
        tc::mbar_arrive_expect_tx(&sm.afull[slot], kARawBytes);
        tc::tma_load_3d(sm.araw[slot], &P.map_a, kQK * (j >> 2) + 64 * (j & 3), tok0, 0, &sm.afull[slot]);
        ++a_next;
        return true;
      };
      auto issue_b = [&]() {
        const int sb = b_next, slot = sb % kBRaw;
        if (!tc::mbar_wait(&sm.bempty[slot], ((sb / kBRaw) & 1) ^ 1, abort_flag)) return false;
        tc::mbar_arrive_expect_tx(&sm.bfull[slot], kBRawBytes);
        tc::tma_load_3d(sm.braw[slot], &P.map_b, 0, row0, sb, &sm.bfull[slot]);
        ++b_next;
        return true;
      };
      auto issue_d8 = [&]() {
        const int sb = d_next, slot = sb & 1;
        if (!tc::mbar_wait(&sm.d8empty[slot], ((sb >> 1) & 1) ^ 1, abort_flag)) return false;
        tc::mbar_arrive_expect_tx(&sm.d8full[slot], kD8RawBytes);
        tc::tma_load_3d(sm.d8raw[slot], &P.map_d8, 32 * sb, tok0, 0, &sm.d8full[slot]);
        ++d_next;
        return true;
      };
      auto issue_s = [&]() {
        const int p = s_next;
        if (!tc::mbar_wait(&sm.sempty, (p & 1) ^ 1, abort_flag)) return false;
        tc::mbar_arrive_expect_tx(&sm.sfull, kSRawBytes);
        tc::tma_load_3d(sm.sraw, &P.map_s, 64 * p, tok0, 0, &sm.sfull);
        ++s_next;
        return true;
      };
      while (ok && a_next < kARaw - 1 && a_next < n_main) ok = issue_a();
      while (ok && b_next < kBRaw - 1 && b_next < nb) ok = issue_b();
      if (ok && with_min) ok = issue_d8();

      int blk = 0, nmin = 0;
      for (int s = 0; s < n_stages && ok; ++s) {
        const StageInfo si = stage_info(s, nb, with_min);
        const int st = s % kStages;
        if (si.kind == 0) {
          // keep kARaw - 1 q8 tiles and kBRaw - 1 superblocks ahead of the
          // converters; each copy goes into the slot freed by the stage just done
          const int j = 4 * si.sb + si.c;
          if (a_next < n_main && a_next <= j + kARaw - 1) ok = issue_a();
          if (ok && si.c == 0 && b_next < nb && b_next <= si.sb + kBRaw - 1) ok = issue_b();
          if (ok && with_min && si.c == 0 && d_next < nb) ok = issue_d8();   // d8 of superblock sb + 1
          if (ok && with_min && si.c == 0 && (si.sb & 1) == 0) ok = issue_s();
          if (!ok) break;
        }
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
      // drain: every MMA issued above completes before TMEM is freed, and
      // every tensor copy issued lands before the CTA exits (after an abort
      // some copies were never consumed)
      tc::mma_commit(&sm.drain);
      bool drained = tc::mbar_wait_sleep(&sm.drain, 0);
      for (int j = a_next - 1; j >= 0 && j >= a_next - kARaw; --j)
        drained &= tc::mbar_wait_sleep(&sm.afull[j % kARaw], (j / kARaw) & 1);
      for (int sb = b_next - 1; sb >= 0 && sb >= b_next - kBRaw; --sb)
        drained &= tc::mbar_wait_sleep(&sm.bfull[sb % kBRaw], (sb / kBRaw) & 1);
      for (int sb = d_next - 1; sb >= 0 && sb >= d_next - 2; --sb)
        drained &= tc::mbar_wait_sleep(&sm.d8full[sb & 1], (sb >> 1) & 1);
      if (s_next > 0) drained &= tc::mbar_wait_sleep(&sm.sfull, (s_next - 1) & 1);
      if (!drained) fail();
    }
  } else if (warp <= kConvWarps) {
    // ------------------------------------------------------------ converters
    // X threads (ci < 96): q8 units ci + 96 i, i < 5 (a unit is 16 int8 of
    // one token: unit u is token u/4, quarter u%4).  Z threads (zi = ci - 96):
    // weight row zi of the tile, plus q8 unit 480 + zi for zi < 32.
    const int ci = threadIdx.x - 32;
    const bool is_z = ci >= kXThreads;
    const int zi = ci - kXThreads;
    const int n_a_units = is_z ? (zi < 32 ? 1 : 0) : 5;
    const int a_unit0 = is_z ? 480 + zi : ci;
    const int a_ustep = is_z ? 0 : kXThreads;
    // header fields kept for the min-term stage, by superblock parity
    uint32_t m03_0 = 0, m47_0 = 0, m03_1 = 0, m47_1 = 0, dmin_0 = 0, dmin_1 = 0, d_bits = 0;
    // token rows of the d8 hand-over and the min-term stage: X threads take
    // tokens ci, the first Z warp tokens 96 + zi
    const bool has_tok = !is_z || zi < 32;
    const int tr = is_z ? 96 + zi : ci;
    uint32_t sc03 = 0x01010101u, sc47 = 0x01010101u;
    bool ok = true;
    for (int s = 0; s < n_stages && ok; ++s) {
      const StageInfo si = stage_info(s, nb, with_min);
      const int st = s % kStages;
      if (si.kind == 0) {
        const int j = 4 * si.sb + si.c;
        const int aslot = j % kARaw, bslot = si.sb % kBRaw;
        const uint8_t* braw_row = sm.braw[bslot] + (is_z ? zi : 0) * kBlockBytes;
        if (is_z && si.c == 0) {
          if (!tc::mbar_wait(&sm.bfull[bslot], (si.sb / kBRaw) & 1, abort_flag)) { ok = false; break; }
          const uint4 h = *reinterpret_cast<const uint4*>(braw_row);
          uint32_t m03, m47;
          header_sc_m(h, sc03, sc47, m03, m47);
          if (dots_only) sc03 = sc47 = 0x01010101u;
          if (si.sb & 1) { m03_1 = m03; m47_1 = m47; dmin_1 = h.x >> 16; }
          else { m03_0 = m03; m47_0 = m47; dmin_0 = h.x >> 16; }
          d_bits = h.x & 0xFFFFu;
        }
        if (with_min && si.c == 0) {
          // hand the epilogue this superblock's d (per row) and d8 (per
          // token, block-major) once it is done with superblock sb - 2
          const int par = si.sb & 1;
          float4 dlo = make_float4(0.f, 0.f, 0.f, 0.f), dhi = dlo;
          if (has_tok) {
            if (!tc::mbar_wait(&sm.d8full[par], (si.sb >> 1) & 1, abort_flag)) { ok = false; break; }
            dlo = *reinterpret_cast<const float4*>(&sm.d8raw[par][tr][0]);
            dhi = *reinterpret_cast<const float4*>(&sm.d8raw[par][tr][4]);
            tc::mbar_arrive(&sm.d8empty[par]);
          }
          if (!tc::mbar_wait(&sm.dempty[par], ((si.sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          if (is_z) sm.dsm[par][zi] = __half2float(__ushort_as_half((unsigned short)d_bits));
          if (has_tok) {
            sm.d8t[par][0][tr] = dlo.x; sm.d8t[par][1][tr] = dlo.y;
            sm.d8t[par][2][tr] = dlo.z; sm.d8t[par][3][tr] = dlo.w;
            sm.d8t[par][4][tr] = dhi.x; sm.d8t[par][5][tr] = dhi.y;
            sm.d8t[par][6][tr] = dhi.z; sm.d8t[par][7][tr] = dhi.w;
          }
          tc::mbar_arrive(&sm.dfull[par]);
        }
        if (!tc::mbar_wait(&sm.afull[aslot], (j / kARaw) & 1, abort_flag)) { ok = false; break; }
        // raw operands to registers
        uint4 av[5];
#pragma unroll
        for (int i = 0; i < 5; ++i)
          if (i < n_a_units)
            av[i] = *reinterpret_cast<const uint4*>(sm.araw[aslot] + 16 * (a_unit0 + a_ustep * i));
        uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
        if (is_z) {
          q0 = *reinterpret_cast<const uint4*>(braw_row + 16 + 32 * si.c);
          q1 = *reinterpret_cast<const uint4*>(braw_row + 32 + 32 * si.c);
        }
        tc::mbar_arrive(&sm.aempty[aslot]);
        if (is_z && si.c == 3) tc::mbar_arrive(&sm.bempty[bslot]);
        if (!tc::mbar_wait(&sm.empty[st], ((s / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
        uint8_t* at = sm.a[st];
        uint8_t* bt = sm.b[st];
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          if (i < n_a_units) {
            const int u = a_unit0 + a_ustep * i;
            const int ar = u >> 2, aq = u & 3;
            uint4 c0, c1;
            cvt_s8x16(av[i], c0, c1);
            *reinterpret_cast<uint4*>(at + tc::sw128_offset(ar, 2 * aq)) = c0;
            *reinterpret_cast<uint4*>(at + tc::sw128_offset(ar, 2 * aq + 1)) = c1;
          }
        }
        if (is_z) {
          // sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)
          const uint32_t scw = si.c < 2 ? sc03 : sc47;
          const uint32_t bsel = 2u * (uint32_t)(si.c & 1);
          const uint32_t slo = byte_h2(scw, bsel), shi = byte_h2(scw, bsel + 1);
          const uint32_t mlo = slo, alo = mul_h2(slo, 0xE400E400u);   // -1024
          const uint32_t mhi = mul_h2(shi, 0x2C002C00u);              // 1/16
          const uint32_t ahi = mul_h2(shi, 0xD400D400u);              // -64
          uint32_t l0, l1, l2, l3, l4, l5, l6, l7, h0, h1, h2, h3, h4, h5, h6, h7;
          cvt_q4x8(q0.x, mlo, alo, mhi, ahi, l0, l1, h0, h1);
          cvt_q4x8(q0.y, mlo, alo, mhi, ahi, l2, l3, h2, h3);
          cvt_q4x8(q0.z, mlo, alo, mhi, ahi, l4, l5, h4, h5);
          cvt_q4x8(q0.w, mlo, alo, mhi, ahi, l6, l7, h6, h7);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 0)) = make_uint4(l0, l1, l2, l3);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 1)) = make_uint4(l4, l5, l6, l7);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 4)) = make_uint4(h0, h1, h2, h3);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 5)) = make_uint4(h4, h5, h6, h7);
          cvt_q4x8(q1.x, mlo, alo, mhi, ahi, l0, l1, h0, h1);
          cvt_q4x8(q1.y, mlo, alo, mhi, ahi, l2, l3, h2, h3);
          cvt_q4x8(q1.z, mlo, alo, mhi, ahi, l4, l5, h4, h5);
          cvt_q4x8(q1.w, mlo, alo, mhi, ahi, l6, l7, h6, h7);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 2)) = make_uint4(l0, l1, l2, l3);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 3)) = make_uint4(l4, l5, l6, l7);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 6)) = make_uint4(h0, h1, h2, h3);
          *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 7)) = make_uint4(h4, h5, h6, h7);
        }
      } else {
        // min-term stage of superblocks 2p, 2p+1: per block, A = (u1,u1,u2,u2)
        // with u = d8*S split into bf16 hi + lo, B = (v1,v2,v1,v2) with
        // v = dmin*m split the same way; the four products sum to u*v.
        const int p = si.sb >> 1;
        if (!tc::mbar_wait(&sm.sfull, p & 1, abort_flag)) { ok = false; break; }
        uint32_t av[32];
        if (has_tok) {
          const int32_t* sp = sm.sraw[tr];
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            // d8 of both superblocks is still in d8t (rewritten only at
            // superblock 2p + 2); a missing second superblock contributes 0
            float u1 = 0.0f, u2 = 0.0f;
            if (b < 8 || si.sb + 1 < nb) split_bf16(sm.d8t[b >> 3][b & 7][tr] * (float)sp[b], u1, u2);
            av[2 * b] = bf16x2(u1, u1);
            av[2 * b + 1] = bf16x2(u2, u2);
          }
        }
        tc::mbar_arrive(&sm.sempty);
        if (!tc::mbar_wait(&sm.empty[st], ((s / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
        uint8_t* at = sm.a[st];
        uint8_t* bt = sm.b[st];
        if (has_tok) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            *reinterpret_cast<uint4*>(at + tc::sw128_offset(tr, jj)) =
                make_uint4(av[4 * jj], av[4 * jj + 1], av[4 * jj + 2], av[4 * jj + 3]);
        }
        if (is_z) {
          const bool row_ok = row0 + zi < rows;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const bool sb_ok = row_ok && si.sb + h < nb;
            const float dmin =
                sb_ok ? __half2float(__ushort_as_half((unsigned short)(h ? dmin_1 : dmin_0))) : 0.0f;
            const uint32_t m03 = h ? m03_1 : m03_0, m47 = h ? m47_1 : m47_0;
            uint32_t bv[16];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
              const uint32_t mv = ((b < 4 ? m03 : m47) >> (8 * (b & 3))) & 0xFFu;
              float v1, v2;
              split_bf16(dmin * (float)mv, v1, v2);
              bv[2 * b] = bf16x2(v1, v2);
              bv[2 * b + 1] = bv[2 * b];
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              *reinterpret_cast<uint4*>(bt + tc::sw128_offset(zi, 4 * h + jj)) =
                  make_uint4(bv[4 * jj], bv[4 * jj + 1], bv[4 * jj + 2], bv[4 * jj + 3]);
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&sm.full[st]);
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
  const int64_t nb = cols / kQK;
  GemmParams P{};
  {
    const uint64_t dims[3] = {(uint64_t)cols, (uint64_t)tokens, 1};
    const uint64_t strides[2] = {(uint64_t)cols, (uint64_t)cols * (uint64_t)tokens};
    const uint32_t box[3] = {64, kBM, 1};
    if (!encode_tmap_u8_3d(&P.map_a, q8, dims, strides, box)) return cudaErrorInvalidValue;
  }
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
  gemm_tc_kernel<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace q4k
