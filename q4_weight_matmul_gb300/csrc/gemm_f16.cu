// q4k_gemm_f16: the prefill GEMM with fp16 activations on the sm_103a tensor
// cores -- the formulation of genie-ai-runtime §3, "The tensor-core kernel
// (Path E)": fp16 operands, fp32 accumulation -- computing the plain product
// of the dequantised weights with fp32 activations,
//
//   y[t][o] = sum_k w[o][k] x[t][k],   w = d*sc*q - dmin*m,
//
// rather than the q8_1 MMQ form of q4k_gemm.
//
// Activations (x_split_f16).  Each token's row is scaled by a power of two
// s_t that puts its largest |x| in [2^14, 2^15), and every scaled element
// X = s_t x is held as two fp16 values, hi = fp16(X) and lo = fp16(X - hi),
// so hi + lo keeps X to 2^-22 of itself (2^-25 absolute below fp16's normal
// range).  The 32-wide block sums XS_b = sum (hi + lo) are kept, times 2^-6,
// as hi/lo fp16 pairs too: per superblock and token 16 values
// [XS_0..XS_7 (hi) | XS_0..XS_7 (lo)].
//
// Weights.  The tensor core reads B = sc*q (an integer <= 945, exact in fp16)
// converted from the BLOCK144 superblocks in shared memory, so the scale
// term of one superblock is one accumulation over its 256 k, hi and lo
// chained into the same fp32 accumulator:
//     acc[t][o] = sum_k (sc*q)[o][k] * (hi + lo)[t][k];
// the min term is one K = 16 MMA against B_min = [m_0..m_7 | m_0..m_7]:
//     macc[t][o] = sum_b m[o][b] * (XS_hi + XS_lo)[t][b];
// and the epilogue adds, once per superblock (not per 32-weight block),
//     total[t][o] += d[o] * acc - 64 * dmin[o] * macc,
// storing y = total / s_t at the end.
//
// Tile: 128 tokens (TMEM lanes) x 128 weight rows (TMEM columns); K walks
// 64 weights per stage, two A tiles (hi, lo) each one tensor copy into the
// 128-byte-swizzled K-major layout; six A tiles (three stages) are in flight
// to cover the copies' latency; one tcgen05.commit per stage releases the
// stage's A and B tiles.  The min-term operands of four consecutive
// superblocks share one tile each (a 32-byte K slot per superblock).  Warp roles in one CTA of 14 warps:
//   warp 0      lane 0 issues every tensor copy: A tiles, one raw 128-row x
//               144-byte superblock tile per superblock, one block-sum tile
//               per four superblocks
//   warp 1      allocates TMEM; lane 0 issues every tcgen05.mma
//   warps 2-5   converters, thread i = weight row i: widen the quants to
//               sc*q fp16, write the row's B_min, hand d and dmin on
//   warps 6-13  epilogue: per superblock, total += d*acc - 64*dmin*macc
// TMEM columns: [0,128) and [128,256) double-buffered superblock
// accumulators, [256,384) the min accumulator, [384,512) the running total.
// The min MMA of superblock sb waits until the epilogue has read superblock
// sb-1's min accumulator, by which time the main MMAs of sb are in flight.
//
// Every mbarrier wait is bounded (tc::kTimeoutCycles); a wait that gives up
// sets the library's device error word, raises a CTA-wide abort flag and the
// CTA unwinds, drains its MMAs and tensor copies and frees its TMEM.
#include "mmq_cvt.cuh"
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

// ------------------------------------------------------------------ split
// One CTA of 256 threads per token row: the row's largest |x| (tree
// reduction), then hi/lo per element and the block sums, one 32-wide block
// per warp iteration (lane k holds element k; the sum is a fixed shuffle tree).
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads) x_split_f16_kernel(const float* __restrict__ x, int64_t cols,
                                                                    __half* __restrict__ hi, __half* __restrict__ lo,
                                                                    __half* __restrict__ bsum,
                                                                    float* __restrict__ inv_scale) {
  __shared__ float red[kSplitThreads / 32];
  __shared__ float s_scale;
  const int64_t t = blockIdx.x;
  const float* xr = x + t * cols;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float amax = 0.0f;
  for (int64_t k = 4 * tid; k < cols; k += 4 * kSplitThreads) {
    const float4 v = *reinterpret_cast<const float4*>(xr + k);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
    for (int i = 1; i < kSplitThreads / 32; ++i) m = fmaxf(m, red[i]);
    // s = 2^(141 - E) for the biased exponent E of the largest |x|, so that
    // s * amax lies in [2^14, 2^15); kept within [2^-126, 2^126] so that 1/s
    // is a normal float too
    const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu);
    const int es = m == 0.0f ? 127 : min(253, max(1, 268 - E));
    const float s = __uint_as_float((uint32_t)es << 23);
    s_scale = s;
    inv_scale[t] = __uint_as_float((uint32_t)(254 - es) << 23);   // 1/s, exact
  }
  __syncthreads();
  const float s = s_scale;
  const int64_t nsub = cols / 32;
  for (int64_t b = warp; b < nsub; b += kSplitThreads / 32) {
    const int64_t k = 32 * b + lane;
    const float X = xr[k] * s;                       // exact: a power of two
    const __half h = __float2half_rn(X);
    const __half l = __float2half_rn(X - __half2float(h));
    hi[t * cols + k] = h;
    lo[t * cols + k] = l;
    float xs = __half2float(h) + __half2float(l);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xs += __shfl_xor_sync(0xffffffffu, xs, o);
    if (lane == 0) {
      const float v = xs * 0.015625f;                // 2^-6: |v| < 2^14
      const __half vh = __float2half_rn(v);
      const __half vl = __float2half_rn(v - __half2float(vh));
      __half* bs = bsum + t * (nsub / 8) * 16 + (b >> 3) * 16 + (b & 7);
      bs[0] = vh;
      bs[8] = vl;
    }
  }
}

// ------------------------------------------------------------------- GEMM
using namespace cvt;

constexpr int kBM = 128;                 // tokens per tile
constexpr int kBN = 128;                 // weight rows per tile
constexpr int kATiles = 6;               // activation tiles in flight (hi, lo of three stages)
constexpr int kBStages = 3;              // fp16 sc*q operand stages (converted)
constexpr int kBRaw = 2;                 // raw superblock tiles in flight
constexpr int kTileBytes = 128 * 128;    // 128 rows x 64 k x fp16
constexpr int kBRawBytes = kBN * kBlockBytes;
constexpr int kConvWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 32 * (2 + kConvWarps + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColMin = 256;
constexpr uint32_t kColTotal = 384;
static_assert(kConvThreads == kBN, "one converter thread per weight row");
static_assert(kATiles == 2 * kBStages, "an A stage (hi, lo) per B stage: one release per stage slot");

struct __align__(1024) Smem {
  uint8_t a[kATiles][kTileBytes];          // fp16 hi / lo activations, 128B-swizzled (tensor copies)
  uint8_t b[kBStages][kTileBytes];         // fp16 sc*q, 128B-swizzled
  uint8_t amin[kTileBytes];                // block sums of four superblocks (tensor copies), 32 bytes each
  uint8_t bmin[kTileBytes];                // [m | m] of superblock sb in 32-byte slot sb % 4
  uint8_t braw[kBRaw][kBRawBytes];         // superblocks as copied
  float dsm[2][kBN];                       // d of each row, by superblock parity
  float dmsm[2][kBN];                      // 64 * dmin of each row
  uint64_t afull[kATiles];
  uint64_t bfull[kBStages];
  uint64_t sempty[kBStages];               // stage slot free: its two A tiles and its B tile
  uint64_t rfull[kBRaw], rempty[kBRaw];
  uint64_t amfull, amempty;
  uint64_t bmfull[4], bmempty[4];
  uint64_t tfull[2], tempty[2];
  uint64_t dfull[2], dempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// 227 KB of dynamic shared memory per CTA, plus the 1024-byte alignment pad
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

struct GemmF16Params {
  CUtensorMap map_hi;   // fp16 {K, tokens}, box {64, 128}, 128-byte swizzle
  CUtensorMap map_lo;
  CUtensorMap map_bs;   // fp16 block sums {16 * nb, tokens}, box {64, 128}, 128-byte swizzle
  CUtensorMap map_b;    // superblocks {144, rows, nb}, box {144, 128, 1}
  const float* inv_scale;
  float* y;
  int* err;
  int rows, nb, tokens;
};

__global__ void __launch_bounds__(kThreads, 1) gemm_f16_kernel(const __grid_constant__ GemmF16Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &sm.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kBN, tok0 = blockIdx.y * kBM;
  const int nb = P.nb, rows = P.rows, tokens = P.tokens;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kATiles; ++i) tc::mbar_init(&sm.afull[i], 1);
    for (int i = 0; i < kBStages; ++i) {
      tc::mbar_init(&sm.bfull[i], kConvThreads);
      tc::mbar_init(&sm.sempty[i], 1);   // one tcgen05.commit per stage releases its A and B tiles
    }
    for (int i = 0; i < kBRaw; ++i) {
      tc::mbar_init(&sm.rfull[i], 1);
      tc::mbar_init(&sm.rempty[i], kConvThreads);
    }
    tc::mbar_init(&sm.amfull, 1);
    tc::mbar_init(&sm.amempty, 1);
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&sm.bmfull[i], kConvThreads);
      tc::mbar_init(&sm.bmempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm.tfull[i], 1);
      tc::mbar_init(&sm.tempty[i], kEpiWarps);
      tc::mbar_init(&sm.dfull[i], kConvThreads);
      tc::mbar_init(&sm.dempty[i], kEpiWarps);
    }
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

  if (warp == 0) {
    // --------------------------------------------------------- tensor copies
    if (lane == 0) {
      bool ok = true;
      int na = 0, nr = 0;           // copies issued
      // The block-sum tile is single: group g is copied as soon as the MMAs
      // of group g-1 are done with it.  Every wait below polls for that
      // (without blocking), so the activation stream never stalls on it.
      const int ngroups = (nb + 3) / 4;
      int gnext = 0;
      auto service = [&]() {
        if (gnext < ngroups && tc::mbar_try_wait(&sm.amempty, (gnext & 1) ^ 1)) {
          tc::mbar_arrive_expect_tx(&sm.amfull, kTileBytes);
          tc::tma_load_2d(sm.amin, &P.map_bs, 64 * gnext, tok0, &sm.amfull);
          ++gnext;
        }
      };
      auto wait_serviced = [&](uint64_t* bar, uint32_t parity) -> bool {
        const long long t0 = clock64();
        for (;;) {
          if (tc::mbar_try_wait(bar, parity)) return true;
          service();
          if (*abort_flag || clock64() - t0 > tc::kTimeoutCycles) return false;
        }
      };
      for (int sb = 0; sb < nb && ok; ++sb) {
        {
          const int slot = sb % kBRaw;
          if (!wait_serviced(&sm.rempty[slot], ((sb / kBRaw) & 1) ^ 1)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.rfull[slot], kBRawBytes);
          tc::tma_load_3d(sm.braw[slot], &P.map_b, 0, row0, sb, &sm.rfull[slot]);
          ++nr;
        }
        service();
        for (int i = 8 * sb; i < 8 * sb + 8; ++i) {   // tile i: stage i/2, hi (even) or lo (odd)
          const int slot = i % kATiles, j = i >> 1;
          if ((i & 1) == 0 && !wait_serviced(&sm.sempty[j % kBStages], ((j / kBStages) & 1) ^ 1)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.afull[slot], kTileBytes);
          tc::tma_load_2d(sm.a[slot], (i & 1) ? &P.map_lo : &P.map_hi, 64 * (i >> 1), tok0, &sm.afull[slot]);
          ++na;
        }
      }
      // the remaining block-sum groups
      while (ok && gnext < ngroups) {
        if (!wait_serviced(&sm.amempty, (gnext & 1) ^ 1)) ok = false;
      }
      const int nm = gnext;
      if (!ok) fail();
      // every copy issued lands before the CTA exits
      bool drained = true;
      for (int i = na - 1; i >= 0 && i >= na - kATiles; --i)
        drained &= tc::mbar_wait_sleep(&sm.afull[i % kATiles], (i / kATiles) & 1);
      for (int sb = nr - 1; sb >= 0 && sb >= nr - kBRaw; --sb)
        drained &= tc::mbar_wait_sleep(&sm.rfull[sb % kBRaw], (sb / kBRaw) & 1);
      if (nm > 0) drained &= tc::mbar_wait_sleep(&sm.amfull, (nm - 1) & 1);
      if (!drained) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idf = tc::idesc_f16(kBM, kBN, false);
      bool ok = true;
      for (int sb = 0; sb < nb && ok; ++sb) {
        const int buf = sb & 1;
        // the epilogue has read this buffer's accumulator (superblock sb - 2)
        if (!tc::mbar_wait(&sm.tempty[buf], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        for (int c = 0; c < 4 && ok; ++c) {
          const int j = 4 * sb + c, sbs = j % kBStages;
          if (!tc::mbar_wait(&sm.bfull[sbs], (j / kBStages) & 1, abort_flag)) { ok = false; break; }
          for (int part = 0; part < 2; ++part) {
            const int i = 2 * j + part, sa = i % kATiles;
            if (!tc::mbar_wait(&sm.afull[sa], (i / kATiles) & 1, abort_flag)) { ok = false; break; }
            tc::fence_after_sync();
            const uint32_t a_base = tc::smem_u32(sm.a[sa]), b_base = tc::smem_u32(sm.b[sbs]);
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_base + 32u * kk), tc::desc_sw128(b_base + 32u * kk),
                             idf, (c | part | kk) ? 1u : 0u);
          }
          if (!ok) break;
          // one release of the stage slot (A tiles and B tile): each
          // tcgen05.commit costs the issuing thread, so one per stage
          tc::mma_commit(&sm.sempty[sbs]);
        }
        if (!ok) break;
        // min term: this superblock's B_min and its group's block sums; the
        // epilogue has read the min accumulator of superblock sb - 1
        const int g = sb >> 2, ms = sb & 3;
        if (!tc::mbar_wait(&sm.bmfull[ms], g & 1, abort_flag) ||
            !tc::mbar_wait(&sm.amfull, g & 1, abort_flag) ||
            (sb > 0 && !tc::mbar_wait(&sm.tempty[buf ^ 1], ((sb - 1) >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        tc::mma_f16_ss(tmem + kColMin, tc::desc_sw128(tc::smem_u32(sm.amin) + 32u * (uint32_t)ms),
                       tc::desc_sw128(tc::smem_u32(sm.bmin) + 32u * (uint32_t)ms), idf, 0u);
        tc::mma_commit(&sm.bmempty[ms]);
        if (ms == 3 || sb == nb - 1) tc::mma_commit(&sm.amempty);
        tc::mma_commit(&sm.tfull[buf]);
      }
      if (!ok) fail();
      // every MMA issued above completes before TMEM is freed
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait_sleep(&sm.drain, 0)) fail();
    }
  } else if (warp < 2 + kConvWarps) {
    // ------------------------------------------------------------ converters
    const int ci = threadIdx.x - 64;             // weight row ci of the tile
    bool ok = true;
    for (int sb = 0; sb < nb && ok; ++sb) {
      const int rslot = sb % kBRaw, par = sb & 1;
      if (!tc::mbar_wait(&sm.rfull[rslot], (sb / kBRaw) & 1, abort_flag)) { ok = false; break; }
      const uint8_t* raw_row = sm.braw[rslot] + ci * kBlockBytes;
      const uint4 hd = *reinterpret_cast<const uint4*>(raw_row);
      uint32_t sc03, sc47, m03, m47;
      header_sc_m(hd, sc03, sc47, m03, m47);
      // B_min row ci: [m_0..m_7 | m_0..m_7] (k 0..15 of the min MMA) in slot sb % 4
      const int ms = sb & 3;
      if (!tc::mbar_wait(&sm.bmempty[ms], ((sb >> 2) & 1) ^ 1, abort_flag)) { ok = false; break; }
      const uint4 mv = make_uint4(bytes_h2(m03, 0, 1), bytes_h2(m03, 2, 3), bytes_h2(m47, 0, 1), bytes_h2(m47, 2, 3));
      *reinterpret_cast<uint4*>(sm.bmin + tc::sw128_offset(ci, 2 * ms)) = mv;
      *reinterpret_cast<uint4*>(sm.bmin + tc::sw128_offset(ci, 2 * ms + 1)) = mv;
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&sm.bmfull[ms]);
      // d and 64*dmin of row ci, once the epilogue is done with superblock sb - 2
      if (!tc::mbar_wait(&sm.dempty[par], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
      sm.dsm[par][ci] = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
      sm.dmsm[par][ci] = 64.0f * __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
      tc::mbar_arrive(&sm.dfull[par]);
      for (int c = 0; c < 4; ++c) {
        const int j = 4 * sb + c, slot = j % kBStages;
        const uint4 q0 = *reinterpret_cast<const uint4*>(raw_row + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(raw_row + 32 + 32 * c);
        if (c == 3) tc::mbar_arrive(&sm.rempty[rslot]);
        if (!tc::mbar_wait(&sm.sempty[slot], ((j / kBStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
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
    }
    if (!ok) fail();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2 - kConvWarps;
    const int q = warp & 3, g = e >> 2;          // TMEM lane quarter (warp % 4), column half
    const int t = 32 * q + lane, tok = tok0 + t;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const int cb = 64 * g;
    bool ok = true;
    for (int sb = 0; sb < nb && ok; ++sb) {
      const int buf = sb & 1;
      // (the TMEM loads below are warp-collective: the warp agrees on the outcome)
      const bool got = tc::mbar_wait(&sm.dfull[buf], (sb >> 1) & 1, abort_flag) &&
                       tc::mbar_wait(&sm.tfull[buf], (sb >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const uint32_t col = (uint32_t)(cb + 16 * qq);
        uint32_t ra[16], rm[16], rt[16];
        tc::tmem_ld16(lane_base + 128u * buf + col, ra);
        tc::tmem_ld16(lane_base + kColMin + col, rm);
        if (sb > 0) {
          tc::tmem_ld16(lane_base + kColTotal + col, rt);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) rt[i] = 0u;
        }
        tc::tmem_wait_ld();
        const float4* dp = reinterpret_cast<const float4*>(&sm.dsm[buf][col]);
        const float4* mp = reinterpret_cast<const float4*>(&sm.dmsm[buf][col]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 dv = dp[i], mv = mp[i];
          const float dd[4] = {dv.x, dv.y, dv.z, dv.w}, dm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int k = 4 * i + u;
            rt[k] = __float_as_uint(fmaf(dd[u], __uint_as_float(ra[k]),
                                         fmaf(-dm[u], __uint_as_float(rm[k]), __uint_as_float(rt[k]))));
          }
        }
        tc::tmem_st16(lane_base + kColTotal + col, rt);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&sm.tempty[buf]);
        tc::mbar_arrive(&sm.dempty[buf]);
      }
    }
    if (ok) {
      // tcgen05.ld is warp-collective: every lane loads, only valid tokens store
      const bool tok_ok = tok < tokens;
      const float inv = tok_ok ? P.inv_scale[tok] : 0.0f;
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        __syncwarp();
        tc::tmem_ld32(lane_base + kColTotal + cb + 32 * half, r);
        tc::tmem_wait_ld();
        const int o0 = row0 + cb + 32 * half;
        if (tok_ok) {
          float* yrow = P.y + (size_t)tok * rows + o0;
          if (o0 + 32 <= rows && (rows & 3) == 0) {
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<float4*>(yrow)[i] =
                  make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                              __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
          } else {
            for (int i = 0; i < 32; ++i)
              if (o0 + i < rows) yrow[i] = __uint_as_float(r[i]) * inv;
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

cudaError_t launch_x_split_f16(const float* x, int64_t tokens, int64_t cols, uint16_t* hi, uint16_t* lo,
                               uint16_t* bsum, float* inv_scale, cudaStream_t s) {
  if (tokens == 0) return cudaSuccess;
  x_split_f16_kernel<<<(unsigned)tokens, kSplitThreads, 0, s>>>(
      x, cols, reinterpret_cast<__half*>(hi), reinterpret_cast<__half*>(lo), reinterpret_cast<__half*>(bsum),
      inv_scale);
  return cudaGetLastError();
}

cudaError_t launch_gemm_f16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                            const uint16_t* bsum, const float* inv_scale, int64_t tokens, float* y, int* err,
                            cudaStream_t s) {
  if (rows == 0 || tokens == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = sizeof(Smem) + 1024;
  static int s_set[64];
  if (!s_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    s_set[dev & 63] = 1;
  }
  const int64_t nb = cols / kQK;
  GemmF16Params P{};
  if (!encode_tmap_2d(&P.map_hi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, hi, (uint64_t)cols, (uint64_t)tokens,
                      (uint64_t)cols * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&P.map_lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, lo, (uint64_t)cols, (uint64_t)tokens,
                      (uint64_t)cols * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&P.map_bs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bsum, (uint64_t)(16 * nb), (uint64_t)tokens,
                      (uint64_t)(32 * nb), 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)kBlockBytes, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)nb * kBlockBytes, (uint64_t)kBlockBytes};
    const uint32_t box[3] = {(uint32_t)kBlockBytes, kBN, 1};
    if (!encode_tmap_u8_3d(&P.map_b, w, dims, strides, box)) return cudaErrorInvalidValue;
  }
  P.inv_scale = inv_scale;
  P.y = y;
  P.err = err;
  P.rows = (int)rows;
  P.nb = (int)nb;
  P.tokens = (int)tokens;
  dim3 grid((unsigned)((rows + kBN - 1) / kBN), (unsigned)((tokens + kBM - 1) / kBM));
  gemm_f16_kernel<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace q4k
