// The decode GEMV kernel behind q4k_gemv, q4k_gemv_multi, q4k_gemv_q8 and
// q6k_gemv: y[b][o] = sum_k w[o][k] x[b][k] (+ residual) over BLOCK144 Q4_K
// (or GPU-layout Q6_K) weights (genie-ai-runtime §4, Path C: packed
// quants read as whole words, dequantised in registers, residual folded in,
// and one kernel for matrices that share their input: the QKV triple and the
// gate/up pair).
//
// Work split.  Rows are cut into blocks of RB rows (RB = 32, 16 or 8: the
// one whose busiest SM costs least, weighing each row by the instructions its
// lanes spend per superblock); one CTA per SM owns a run of
// row blocks (of one or several matrices) and all their superblocks.  A unit
// of work is one row block x one superblock; the 15 consumer warps take units
// round-robin, so K is split across warps.  Each unit leaves one partial sum
// per row in shared memory and the CTA adds a row's partials in superblock
// order (bitwise deterministic).
//
// Streaming.  A producer warp fetches the weights with 3-D tensor copies:
// one copy per stage of RB rows x (128/RB) superblocks (18 KB, out-of-range
// rows and superblocks zero-filled) into a ring of stages.  The copies start
// at launch, before the activations are read.  The ring is as deep as
// shared memory allows (up to 6 stages); launched as a programmatic dependent
// (opt-in, see pdl_mode) the CTA first keeps under ~110 KB so that the next
// GEMV's CTA can start on its SM, and griddepcontrol.wait orders every
// activation read after the previous kernel has completed.
//
// Lanes.  32/RB lanes share a row: with RB = 32 a lane owns a row's whole
// superblock (256 weights), with RB = 16 half of it, with RB = 8 one 64-weight
// chunk.  A chunk's 32 quant bytes hold sub-block 2c in low nibbles and 2c+1
// in high nibbles.
//
// Arithmetic: 32-bit fixed-point activation digit planes and exact integer
// dp4a block sums, scales applied in fp32 (gemv_common.cuh).
//
// q8_1 activations (q4k_gemv_q8, and q4k_gemm for a few tokens): the same
// kernel with the activation kind a template parameter; the quants are
// staged as one int8 plane and the block dots are the exact integer MMQ dots.
//
// Q6_K weights (q6k_gemv): the same kernel with the weight format a template
// parameter.  The GPU layout (q6k_pack.cu) puts a row's 208-byte superblocks
// (scales and quants) and its d values in separate regions, so a stage is two
// tensor copies: RB rows x SB superblocks of 208 bytes, and RB rows x 8 d
// values (16 bytes, the aligned group of 8 that holds the stage's SB).
#pragma once

#include "gemv_common.cuh"
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

constexpr int kConsumerWarps = 15;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;     // + one producer warp
constexpr int kStageSuper = 128;              // superblock-rows per stage (RB * SB)
constexpr int kMaxRing = 6;
constexpr size_t kPairSmem = 110 * 1024;      // a CTA this small leaves room for a neighbour
constexpr int kMaxMats = 4;

// weight formats
constexpr int kFmtQ4K = 0;      // BLOCK144 Q4_K
constexpr int kFmtQ6K = 1;      // Q6_K, GPU layout

// per format: bytes of a superblock, superblock-rows per stage, bytes of a
// stage (for Q6_K the d box, at most 32 rows x 8 values, follows the blocks)
template <int FMT> struct Fmt;
template <> struct Fmt<kFmtQ4K> {
  static constexpr int kBlk = kBlockBytes, kSuper = kStageSuper, kDBytes = 0;
  static constexpr int kStage = kSuper * kBlk;
};
template <> struct Fmt<kFmtQ6K> {
  static constexpr int kBlk = gemv::kQ6Blk, kSuper = 64, kDBytes = 32 * 16;
  static constexpr int kStage = kSuper * kBlk + kDBytes;
};
static_assert(Fmt<kFmtQ6K>::kStage % 128 == 0 && (Fmt<kFmtQ6K>::kSuper * gemv::kQ6Blk) % 128 == 0,
              "tensor-copy destinations stay 128-byte aligned");

struct GemvParams {
  CUtensorMap map[kMaxMats];
  CUtensorMap dmap[kMaxMats];   // Q6_K: the d values of each row
  float* y[kMaxMats];
  const float* res[kMaxMats];
  int rows[kMaxMats];
  int rb_start[kMaxMats + 1];   // prefix sums of row blocks per matrix
  int n_mats;
  int nb, rb_per_cta, rb_pass, ring;
  int pdl;                      // launched as a programmatic dependent
  int trigger_late;             // launch dependents after the units, not at start
  const float* x;
  const void* xq;               // q8_1 quants (int8, or binary16 integers)
  const float* d8;
  const int32_t* qsum;
  int32_t* p_out;               // non-null: store the q8 block dots too (one matrix)
  int* err;
};

// activation kinds
constexpr int kActF32 = 0;      // fp32 x, fixed-point digit planes
constexpr int kActQ8 = 1;       // q8_1, int8 quants
constexpr int kActQ8H = 2;      // q8_1, binary16 quants

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

struct Layout {
  size_t xs, xsum, part, stages, bars, total;
};

__host__ __device__ inline Layout layout(int B, int nb, int ring, int part_floats, bool q8, int stage_bytes) {
  Layout L;
  L.xs = 0;
  L.xsum = L.xs + (q8 ? gemv::xq8_bytes(B, nb) : gemv::xs_bytes(B, nb));
  L.part = L.xsum + (q8 ? gemv::xq8s_bytes(B, nb) : gemv::xss_bytes(B, nb));
  L.stages = (L.part + sizeof(float) * (size_t)part_floats + 1023) & ~size_t(1023);
  L.bars = L.stages + (size_t)ring * stage_bytes;
  L.total = L.bars + sizeof(uint64_t) * 2 * ring + 16 + 1024;   // + issue counter, + slack to align the base
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

// LPR: lanes per row (1, 2 or 4); RB = 32 / LPR rows per block.  ACT: the
// activation kind.  FMT: the weight format.
template <int B, int LPR, int ACT, int FMT>
__global__ void __launch_bounds__(kThreads, 1) gemv_block144_kernel(
    const __grid_constant__ GemvParams P) {
  constexpr int RB = 32 / LPR;              // rows per block
  constexpr int kBlk = Fmt<FMT>::kBlk;
  constexpr int kStageBytes = Fmt<FMT>::kStage;
  constexpr int SB = Fmt<FMT>::kSuper / RB; // superblocks per stage
  constexpr int kTx = Fmt<FMT>::kSuper * kBlk + (FMT == kFmtQ6K ? RB * 16 : 0);   // bytes a stage receives
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
  const Layout L = layout(B, nb, ring, B * rb_pass * nb * RB, ACT != kActF32, kStageBytes);
  uint8_t* xs = smem + L.xs;
  float2* xss = reinterpret_cast<float2*>(smem + L.xsum);
  float* part = reinterpret_cast<float*>(smem + L.part);      // [B][rb of the pass][nb][RB]
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ring;
  volatile int* issued = reinterpret_cast<volatile int*>(empty + ring);   // stages issued so far
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // the next kernel in the stream may start its own weight stream now
  if (P.pdl && !P.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < ring; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], SB);
    }
    *issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int slot = 0, g = rb0, sj = 0;
      int m = mat_of(P, g);
      uint32_t phase = 0;
      int n_issued = 0;
      for (int j = 0; j < n_stages; ++j) {
        if (!tc::mbar_wait_sleep(&empty[slot], phase ^ 1)) {
          atomicOr(P.err, 2);
          break;
        }
        ++n_issued;
        tc::mbar_arrive_expect_tx(&full[slot], kTx);
        tc::tma_load_3d(stages + (size_t)slot * kStageBytes, &P.map[m], 0, (g - P.rb_start[m]) * RB, sj * SB,
                        &full[slot]);
        if constexpr (FMT == kFmtQ6K)   // d: the aligned group of 8 superblocks holding this stage's SB
          tc::tma_load_2d(stages + (size_t)slot * kStageBytes + Fmt<FMT>::kSuper * kBlk, &P.dmap[m],
                          (sj * SB) & ~7, (g - P.rb_start[m]) * RB, &full[slot]);
        __threadfence_block();
        *issued = j + 1;
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
      for (int j = max(0, n_issued - ring); j < n_issued; ++j)
        if (!tc::mbar_wait_sleep(&full[j % ring], (uint32_t)((j / ring) & 1))) atomicOr(P.err, 2);
    }
    if (P.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }

  // -------------------------------------------------------------- consumers
  if (P.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (ACT == kActF32) gemv::stage_x<B, kConsumers, false>(P.x, nb, xs, xss, tid);
  else gemv::stage_q8<B, kConsumers, ACT == kActQ8H>(P.xq, P.d8, P.qsum, nb, xs, xss, tid);
  named_sync_consumers();
  const gemv::XView xv = gemv::make_view(xs, xss, P.x, B, nb);

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
      // A warp only takes its own units, so it may reach stage j while the
      // copy of stage j - ring (same slot, same parity two phases back) is
      // still in flight; the parity wait is unambiguous only once the
      // producer has issued stage j, which it does after stage j - ring
      // has landed and been consumed.
      if (ok && *issued <= j && !gemv::wait_issued(issued, j)) {
        ok = false;
        if (lane == 0) atomicOr(P.err, 2);
      }
      if (ok && !tc::mbar_wait_sleep(&full[slot], phase)) {
        ok = false;
        if (lane == 0) atomicOr(P.err, 2);
      }
      float acc[B];
#pragma unroll
      for (int b = 0; b < B; ++b) acc[b] = 0.0f;
      if (sb < nb) {
        // stage laid out [SB][RB][kBlk] (rows inner), then (Q6_K) d as [RB][8]
        const uint8_t* p = stages + (size_t)slot * kStageBytes + ((size_t)z * RB + r_in) * kBlk;
        if constexpr (FMT == kFmtQ6K) {
          const __half* dv = reinterpret_cast<const __half*>(stages + (size_t)slot * kStageBytes +
                                                             Fmt<FMT>::kSuper * kBlk);
          const float dd = __half2float(dv[r_in * 8 + ((sj * SB) & 7) + z]);
          if constexpr (ACT == kActF32) {
            gemv::superblock_dot_q6<B, CPL, false>(p, dd, xv, sb, c0, acc);
          } else {
            int32_t* pout = nullptr;
            if (P.p_out) {
              const int row = (rb0 + pb + rbl - P.rb_start[0]) * RB + r_in;
              if (row < P.rows[0]) pout = P.p_out + ((size_t)row * nb + sb) * 16;
            }
            gemv::superblock_dot_q6_q8<B, CPL>(p, dd, xs, xss, nb, sb, c0, acc, pout, (size_t)P.rows[0] * nb * 16);
          }
        } else if constexpr (ACT == kActF32) {
          gemv::superblock_dot<B, CPL, false>(p, xv, sb, c0, acc);
        } else {
          int32_t* pout = nullptr;
          if (P.p_out) {
            const int g = rb0 + pb + rbl;
            const int row = (g - P.rb_start[0]) * RB + r_in;
            if (row < P.rows[0]) pout = P.p_out + ((size_t)row * nb + sb) * 8;
          }
          gemv::superblock_dot_q8<B, CPL>(p, xs, xss, nb, sb, c0, acc, pout, (size_t)P.rows[0] * nb * 8);
        }
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
      if (row < rows && ok && P.y[m]) {   // (no y when only the block dots are wanted)
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

Plan make_plan(int B, const int64_t* rows, int n_mats, int nb, const DeviceInfo& info, bool q8, int fmt) {
  const int stage_bytes = fmt == kFmtQ6K ? Fmt<kFmtQ6K>::kStage : Fmt<kFmtQ4K>::kStage;
  Plan p{};
  // rows per block: the choice whose busiest SM costs least, a row costing
  // the instructions its lanes spend per superblock -- a lane that owns a whole
  // superblock (32-row blocks) pays the per-unit costs (waits, scale decode,
  // partial store, activation loads) once per 256 weights, a quarter-superblock
  // lane once per 64 (measured: ~1.8x the instructions per weight with 8-row
  // blocks, ~1.35x with 16-row blocks)
  constexpr int64_t kCost[3] = {20, 27, 36};   // per row, 32-, 16-, 8-row blocks
  int64_t best = INT64_MAX;
  p.lpr = 1;
  for (int i = 0; i < 3; ++i) {
    const int64_t rb = 32 >> i;
    int64_t n_rb = 0;
    for (int m = 0; m < n_mats; ++m) n_rb += (rows[m] + rb - 1) / rb;
    const int64_t cost = (n_rb + info.sm_count - 1) / info.sm_count * rb * kCost[i];
    if (cost < best) {
      best = cost;
      p.lpr = 1 << i;
    }
  }
  const int RB = 32 / p.lpr;
  int64_t n_rb = 0;
  for (int m = 0; m < n_mats; ++m) n_rb += (rows[m] + RB - 1) / RB;
  p.rb_per_cta = (int)((n_rb + info.sm_count - 1) / info.sm_count);
  p.grid = (int)((n_rb + p.rb_per_cta - 1) / p.rb_per_cta);
  // partial sums of at most 8 KB per pass
  p.rb_pass = (int)std::max<int64_t>(1, std::min<int64_t>(p.rb_per_cta, 2048 / ((int64_t)B * nb * RB)));
  // the deepest ring that fits; launched as a programmatic dependent (opt-in),
  // first the deepest that keeps the CTA small enough to share its SM with
  // the next kernel's
  p.ring = 0;
  const size_t caps[2] = {pdl_mode() != 0 ? kPairSmem : (size_t)info.max_smem_optin, (size_t)info.max_smem_optin};
  for (size_t cap : caps) {
    for (int ring = kMaxRing; ring >= 2 && p.ring == 0; --ring) {
      const size_t total = layout(B, nb, ring, B * p.rb_pass * nb * RB, q8, stage_bytes).total;
      if (total <= cap) {
        p.ring = ring;
        p.smem = total;
      }
    }
    if (p.ring) break;
  }
  return p;
}

template <int B, int LPR, int ACT, int FMT>
cudaError_t launch_bl(const GemvParams& params, const Plan& p, int dev, const DeviceInfo& info,
                      cudaStream_t s) {
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if (limit < info.max_smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_block144_kernel<B, LPR, ACT, FMT>,
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
  return cudaLaunchKernelEx(&cfg, gemv_block144_kernel<B, LPR, ACT, FMT>, params);
}

struct ActIn {   // the activations of one launch
  const float* x;
  const void* xq;
  const float* d8;
  const int32_t* qsum;
  int32_t* p_out;
};

template <int B, int ACT, int FMT>
cudaError_t launch_b(const uint8_t* const* w, const int64_t* rows, int n_mats, int nb, const ActIn& act,
                     const float* const* residual, float* const* y, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo& info = device_info(dev);
  const Plan p = make_plan(B, rows, n_mats, nb, info, ACT != kActF32, FMT);
  if (p.ring == 0) return cudaErrorNotSupported;
  GemvParams params;
  memset(&params, 0, sizeof(params));
  params.err = device_error_word();
  if (!params.err) return cudaErrorInvalidValue;
  constexpr bool q6 = FMT == kFmtQ6K;
  const int RB = 32 / p.lpr, SB = (q6 ? Fmt<kFmtQ6K>::kSuper : Fmt<kFmtQ4K>::kSuper) / RB;
  const uint64_t blk = q6 ? (uint64_t)gemv::kQ6Blk : (uint64_t)kBlockBytes;
  const uint64_t row_bytes = q6 ? (uint64_t)q6k_gpu_row_bytes(nb) : (uint64_t)nb * kBlockBytes;
  params.n_mats = n_mats;
  params.rb_start[0] = 0;
  for (int m = 0; m < n_mats; ++m) {
    // box: a superblock's bytes x RB rows x SB superblocks, rows inner in shared memory
    const uint64_t dims[3] = {blk, (uint64_t)rows[m], (uint64_t)nb};
    const uint64_t strides[2] = {row_bytes, blk};
    const uint32_t box[3] = {(uint32_t)blk, (uint32_t)RB, (uint32_t)SB};
    if (!encode_tmap_u8_3d(&params.map[m], w[m], dims, strides, box)) return cudaErrorInvalidValue;
    // Q6_K: the row's d values follow its superblocks; box 8 values x RB rows
    if (q6 && !encode_tmap_2d(&params.dmap[m], CU_TENSOR_MAP_DATA_TYPE_UINT16, w[m] + (size_t)nb * blk,
                              (uint64_t)nb, (uint64_t)rows[m], row_bytes, 8, (uint32_t)RB,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
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
  params.pdl = pdl_mode() != 0 ? 1 : 0;
  params.trigger_late = pdl_mode() == 2 ? 1 : 0;
  params.x = act.x;
  params.xq = act.xq;
  params.d8 = act.d8;
  params.qsum = act.qsum;
  params.p_out = act.p_out;
  switch (p.lpr) {
    case 1: return launch_bl<B, 1, ACT, FMT>(params, p, dev, info, s);
    case 2: return launch_bl<B, 2, ACT, FMT>(params, p, dev, info, s);
    default: return launch_bl<B, 4, ACT, FMT>(params, p, dev, info, s);
  }
}

// Launch of one activation kind ACT and weight format FMT; each translation
// unit that calls it instantiates the kernels of its own kinds only.
template <int ACT, int FMT>
cudaError_t launch_batch(const uint8_t* const* w, const int64_t* rows, int n_mats, int nb, int batch,
                         const ActIn& act, const float* const* residual, float* const* y, cudaStream_t s) {
  switch (batch) {
    case 1: return launch_b<1, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 2: return launch_b<2, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 3: return launch_b<3, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 4: return launch_b<4, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 5: return launch_b<5, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 6: return launch_b<6, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 7: return launch_b<7, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    case 8: return launch_b<8, ACT, FMT>(w, rows, n_mats, nb, act, residual, y, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace
}  // namespace q4k
