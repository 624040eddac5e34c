// q6k_gemm_f16: the fp16-activation prefill GEMM of gemm_f16.cu over Q6_K
// weights in the GPU layout (genie-ai-runtime §3, "The tensor-core kernel
// (Path E)" for the Q6_K half of Q4_K_M):
//
//   y[t][o] = sum_k w[o][k] x[t][k],   w = d * sc_g * (q - 32),
//
// with the activations split by x_split_f16 (per-token power-of-two scale,
// hi/lo fp16).  The weight operand of a 16-weight group is v = sc*(q - 32),
// an integer in [-4096, 4064]: fp16 holds it exactly only up to 2048, so it
// is carried as B_hi = fp16(v) and B_lo = v - B_hi (-1, 0 or 1), both exact,
// formed with one fp16 multiply and one fp16 FMA from the exact fp16 value
// 4*(q - 32) and sc/4.  Each K slice takes three MMAs into the superblock's
// fp32 accumulator: hi*B_hi + lo*B_hi + hi*B_lo (the dropped lo*B_lo is below
// 2^-22 of the product).  There is no min term; the epilogue adds d * acc into
// the running total once per superblock.
//
// Tile 128 tokens x 128 weight rows, K in 64-wide stages (one 48-byte chunk
// of each superblock row).  Roles as in gemm_f16.cu: warp 0 issues the
// tensor copies (activation tiles; per superblock one 128-row x 208-byte box
// and one 128-row box of the rows' d values), warp 1 allocates TMEM and
// issues the MMAs, warps 2-5 convert (thread i = weight row i), warps 6-13
// run the epilogue.  TMEM: [0,256) double-buffered superblock accumulators,
// [256,384) the running total.  One tcgen05.commit per stage releases the
// stage's A tiles and its two B tiles.  Every wait is bounded.
#include "gemv_common.cuh"
#include "mmq_cvt.cuh"
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

namespace q4k {
namespace {

constexpr int kBM = 128;                 // tokens per tile
constexpr int kBN = 128;                 // weight rows per tile
constexpr int kBStages = 2;              // converted stages (B_hi and B_lo tiles each)
constexpr int kATiles = 2 * kBStages;    // activation tiles (hi, lo of each stage)
constexpr int kBRaw = 2;                 // raw superblock tiles in flight
constexpr int kTileBytes = 128 * 128;    // 128 rows x 64 k x fp16
constexpr int kRawBytes = kBN * gemv::kQ6Blk;
constexpr int kDRawBytes = kBN * 16;     // 128 rows x 8 binary16 d values
constexpr int kConvWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 32 * (2 + kConvWarps + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColTotal = 256;
static_assert(kConvThreads == kBN, "one converter thread per weight row");

struct __align__(1024) Smem {
  uint8_t a[kATiles][kTileBytes];          // fp16 hi / lo activations, 128B-swizzled (tensor copies)
  uint8_t b[kBStages][2][kTileBytes];      // B_hi, B_lo, 128B-swizzled
  uint8_t braw[kBRaw][kRawBytes];          // Q6_K superblocks as copied
  uint16_t draw[kBRaw][kBN * 8];           // binary16 d of an aligned group of 8 superblocks, per row
  float dsm[2][kBN];                       // d of each row, by superblock parity
  uint64_t afull[kATiles];
  uint64_t bfull[kBStages];
  uint64_t sempty[kBStages];               // stage slot free: its A tiles and its B tiles
  uint64_t rfull[kBRaw], rempty[kBRaw];
  uint64_t tfull[2], tempty[2];
  uint64_t dfull[2], dempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");

struct GemmQ6Params {
  CUtensorMap map_hi;   // fp16 {K, tokens}, box {64, 128}, 128-byte swizzle
  CUtensorMap map_lo;
  CUtensorMap map_b;    // superblocks {208, rows, nb}, box {208, 128, 1}
  CUtensorMap map_d;    // d values {nb, rows} (binary16), box {8, 128}
  const float* inv_scale;
  float* y;
  int* err;
  int rows, nb, tokens;
};

// B_hi, B_lo fp16x2 pairs of the four signed bytes 4*(q - 32) in w (two
// pairs each, k order), for a group scale whose sc/4 is sc4 (fp16x2)
__device__ __forceinline__ void cvt_q6x4(uint32_t w, uint32_t sc4, uint32_t& hi01, uint32_t& hi23,
                                         uint32_t& lo01, uint32_t& lo23) {
  const uint32_t u = w ^ 0x80808080u;                           // 4*(q - 32) + 128, unsigned bytes
  uint32_t f01, f23;
  asm("{\n\t.reg .b32 t01, t23, z, k;\n\tmov.b32 z, 0;\n\tmov.b32 k, 0x64806480;\n\t"   // k = 1024 + 128
      "prmt.b32 t01, %2, z, 0x4140;\n\tprmt.b32 t23, %2, z, 0x4342;\n\t"
      "or.b32 t01, t01, 0x64006400;\n\tor.b32 t23, t23, 0x64006400;\n\t"
      "sub.rn.f16x2 %0, t01, k;\n\tsub.rn.f16x2 %1, t23, k;\n\t}"
      : "=r"(f01), "=r"(f23) : "r"(u));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi01) : "r"(f01), "r"(sc4));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi23) : "r"(f23), "r"(sc4));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo01) : "r"(f01), "r"(sc4), "r"(hi01 ^ 0x80008000u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo23) : "r"(f23), "r"(sc4), "r"(hi23 ^ 0x80008000u));
}

// fp16x2 (sc/4, sc/4) of the signed scale byte `bi` of word w (exact)
__device__ __forceinline__ uint32_t scale4_h2(uint32_t w, int bi) {
  const float v = 0.25f * (float)(int8_t)((w >> (8 * bi)) & 0xFFu);
  const __half h = __float2half_rn(v);
  const uint32_t b = (uint32_t)__half_as_ushort(h);
  return b | (b << 16);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_q6k_f16_kernel(const __grid_constant__ GemmQ6Params P) {
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
      tc::mbar_init(&sm.sempty[i], 1);
    }
    for (int i = 0; i < kBRaw; ++i) {
      tc::mbar_init(&sm.rfull[i], 1);
      tc::mbar_init(&sm.rempty[i], kConvThreads);
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
      int na = 0, nr = 0;
      for (int sb = 0; sb < nb && ok; ++sb) {
        {
          const int slot = sb % kBRaw;
          if (!tc::mbar_wait(&sm.rempty[slot], ((sb / kBRaw) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.rfull[slot], kRawBytes + kDRawBytes);
          tc::tma_load_3d(sm.braw[slot], &P.map_b, 0, row0, sb, &sm.rfull[slot]);
          tc::tma_load_2d(sm.draw[slot], &P.map_d, sb & ~7, row0, &sm.rfull[slot]);
          ++nr;
        }
        for (int i = 8 * sb; i < 8 * sb + 8; ++i) {   // tile i: stage i/2, hi (even) or lo (odd)
          const int slot = i % kATiles, j = i >> 1;
          if ((i & 1) == 0 && !tc::mbar_wait(&sm.sempty[j % kBStages], ((j / kBStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&sm.afull[slot], kTileBytes);
          tc::tma_load_2d(sm.a[slot], (i & 1) ? &P.map_lo : &P.map_hi, 64 * j, tok0, &sm.afull[slot]);
          ++na;
        }
      }
      if (!ok) fail();
      bool drained = true;
      for (int i = na - 1; i >= 0 && i >= na - kATiles; --i)
        drained &= tc::mbar_wait_sleep(&sm.afull[i % kATiles], (i / kATiles) & 1);
      for (int sb = nr - 1; sb >= 0 && sb >= nr - kBRaw; --sb)
        drained &= tc::mbar_wait_sleep(&sm.rfull[sb % kBRaw], (sb / kBRaw) & 1);
      if (!drained) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idf = tc::idesc_f16(kBM, kBN, false);
      bool ok = true;
      for (int sb = 0; sb < nb && ok; ++sb) {
        const int buf = sb & 1;
        if (!tc::mbar_wait(&sm.tempty[buf], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        for (int c = 0; c < 4 && ok; ++c) {
          const int j = 4 * sb + c, sbs = j % kBStages;
          const int ih = (2 * j) % kATiles, il = (2 * j + 1) % kATiles;
          if (!tc::mbar_wait(&sm.bfull[sbs], (j / kBStages) & 1, abort_flag) ||
              !tc::mbar_wait(&sm.afull[ih], ((2 * j) / kATiles) & 1, abort_flag) ||
              !tc::mbar_wait(&sm.afull[il], ((2 * j + 1) / kATiles) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_hi = tc::smem_u32(sm.a[ih]), a_lo = tc::smem_u32(sm.a[il]);
          const uint32_t b_hi = tc::smem_u32(sm.b[sbs][0]), b_lo = tc::smem_u32(sm.b[sbs][1]);
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t ko = 32u * kk;
            tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_hi + ko), tc::desc_sw128(b_hi + ko), idf,
                           (c | kk) ? 1u : 0u);
            tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_lo + ko), tc::desc_sw128(b_hi + ko), idf, 1u);
            tc::mma_f16_ss(tmem + 128u * buf, tc::desc_sw128(a_hi + ko), tc::desc_sw128(b_lo + ko), idf, 1u);
          }
          // one release of the stage slot (A tiles, B tiles)
          tc::mma_commit(&sm.sempty[sbs]);
        }
        if (!ok) break;
        tc::mma_commit(&sm.tfull[buf]);
      }
      if (!ok) fail();
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
      const uint8_t* raw_row = sm.braw[rslot] + ci * gemv::kQ6Blk;
      const uint4 scv = *reinterpret_cast<const uint4*>(raw_row);
      const float d = __half2float(__ushort_as_half(sm.draw[rslot][ci * 8 + (sb & 7)]));
      // d of row ci, once the epilogue is done with superblock sb - 2
      if (!tc::mbar_wait(&sm.dempty[par], ((sb >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
      sm.dsm[par][ci] = d;
      tc::mbar_arrive(&sm.dfull[par]);
      for (int c = 0; c < 4; ++c) {
        const int j = 4 * sb + c, slot = j % kBStages;
        const uint8_t* ch = raw_row + 16 + 48 * c;
        const uint4 l0 = *reinterpret_cast<const uint4*>(ch);
        const uint4 l1 = *reinterpret_cast<const uint4*>(ch + 16);
        const uint4 hw = *reinterpret_cast<const uint4*>(ch + 32);
        if (c == 3) tc::mbar_arrive(&sm.rempty[rslot]);
        if (!tc::mbar_wait(&sm.sempty[slot], ((j / kBStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
        uint8_t* bh = sm.b[slot][0];
        uint8_t* bl = sm.b[slot][1];
        const uint32_t scw = gemv::word_of(scv, c);   // groups 4c + 2s + h
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 lv = h ? l1 : l0;
            const uint32_t sc4 = scale4_h2(scw, 2 * s2 + h);
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t w = gemv::q6_word(gemv::word_of(lv, k), gemv::word_of(hw, k), s2, h);
              cvt_q6x4(w, sc4, hi[2 * k], hi[2 * k + 1], lo[2 * k], lo[2 * k + 1]);
            }
            // k = 32 s2 + 16 h + 4 kw + i: 16-byte chunks 4 s2 + 2 h and 4 s2 + 2 h + 1
            const int c0 = 4 * s2 + 2 * h;
            *reinterpret_cast<uint4*>(bh + tc::sw128_offset(ci, c0)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(bh + tc::sw128_offset(ci, c0 + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
            *reinterpret_cast<uint4*>(bl + tc::sw128_offset(ci, c0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4*>(bl + tc::sw128_offset(ci, c0 + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
          }
        }
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
        uint32_t ra[16], rt[16];
        tc::tmem_ld16(lane_base + 128u * buf + col, ra);
        if (sb > 0) {
          tc::tmem_ld16(lane_base + kColTotal + col, rt);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) rt[i] = 0u;
        }
        tc::tmem_wait_ld();
        const float4* dp = reinterpret_cast<const float4*>(&sm.dsm[buf][col]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 dv = dp[i];
          const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            rt[4 * i + u] = __float_as_uint(fmaf(dd[u], __uint_as_float(ra[4 * i + u]), __uint_as_float(rt[4 * i + u])));
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

cudaError_t launch_gemm_q6k_f16(const uint8_t* w, int64_t rows, int64_t cols, const uint16_t* hi, const uint16_t* lo,
                                const float* inv_scale, int64_t tokens, float* y, int* err, cudaStream_t s) {
  if (rows == 0 || tokens == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = sizeof(Smem) + 1024;
  static int s_set[64];
  if (!s_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_q6k_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    s_set[dev & 63] = 1;
  }
  const int64_t nb = cols / kQK;
  const uint64_t row_bytes = (uint64_t)q6k_gpu_row_bytes(nb);
  GemmQ6Params P{};
  if (!encode_tmap_2d(&P.map_hi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, hi, (uint64_t)cols, (uint64_t)tokens,
                      (uint64_t)cols * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&P.map_lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, lo, (uint64_t)cols, (uint64_t)tokens,
                      (uint64_t)cols * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&P.map_d, CU_TENSOR_MAP_DATA_TYPE_UINT16, w + (size_t)nb * gemv::kQ6Blk, (uint64_t)nb,
                      (uint64_t)rows, row_bytes, 8, kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)gemv::kQ6Blk, (uint64_t)rows, (uint64_t)nb};
    const uint64_t strides[2] = {row_bytes, (uint64_t)gemv::kQ6Blk};
    const uint32_t box[3] = {(uint32_t)gemv::kQ6Blk, kBN, 1};
    if (!encode_tmap_u8_3d(&P.map_b, w, dims, strides, box)) return cudaErrorInvalidValue;
  }
  P.inv_scale = inv_scale;
  P.y = y;
  P.err = err;
  P.rows = (int)rows;
  P.nb = (int)nb;
  P.tokens = (int)tokens;
  dim3 grid((unsigned)((rows + kBN - 1) / kBN), (unsigned)((tokens + kBM - 1) / kBM));
  gemm_q6k_f16_kernel<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace q4k
