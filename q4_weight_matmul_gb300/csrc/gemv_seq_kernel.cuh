// The persistent job-list GEMV kernel of q4k_gemv_seq (host side in
// gemv_seq.cu): an ordered list of decode GEMV jobs y = W x (+ residual) over
// BLOCK144 Q4_K (or GPU-layout Q6_K) weights in one persistent launch (genie-ai-runtime §4,
// Path C: the GEMVs are the hot decode kernels and every decode step streams
// the whole model; §2: decode is bound by memory bandwidth).
//
// One CTA per SM stays resident for the whole list.  Its producer thread
// streams weights into a shared-memory ring with 3-D tensor copies and waits
// for nothing but a free slot, so the weight stream runs on across matrix
// boundaries and across the dependency points between jobs; 15 consumer
// warps dequantise and reduce.  This removes the launch gap, the start-up
// latency and the drain that separate launches pay at every matrix boundary.
//
// Segments and epochs.  Consecutive jobs that read the same x (same cols)
// form a segment; the segments between two jobs with `wait` set form an
// epoch.  An epoch reads its activations only after every earlier job has
// completed (a grid-wide arrival counter in the workspace); that is how a job
// consumes an earlier job's output inside the launch.  Only the activation
// reads wait: the weights of the waiting epoch are already streaming into
// the ring.
//
// Units.  Rows are cut into blocks of 32; a unit is one row block x two
// superblocks (32 x 2 x 144 bytes) and is one tensor copy into one ring slot,
// laid out [superblock][row][144] so that lane r of the consuming warp reads
// row r without bank conflicts and all 32 lanes read the same activations
// (broadcast).  On GB300 a tensor copy costs the copy engine a roughly fixed
// time: boxes of 4.6 KB stream at about half the HBM rate, boxes of 9 KB and
// more at nearly all of it.
//
// Work split.  An epoch's units (its segments in order, each
// row-block-major) are cut into equal contiguous ranges, one per CTA, so
// every SM streams the same number of bytes whatever the matrix shapes, and
// a CTA stages new activations only where its range enters another segment.
// A row block cut by range boundaries is finished by several CTAs: each
// stores its partial row sums in the workspace and the last one to finish
// adds the pieces in CTA order (the result does not depend on timing) and
// stores y.  For a small epoch, where that final combine would cost more
// than the imbalance, the range boundaries move back to row-block starts
// instead (choose_aligned).  A launch takes up to 96 jobs, 48 of them Q6_K
// (their tensor maps travel in the kernel parameters); longer lists take
// several launches.
//
// Q6_K jobs (GPU layout) are units of 32 rows x 2 superblocks of 208 bytes
// plus the rows' d values (a second tensor copy); a segment holds one format,
// and a launch that holds a Q6_K job sizes every ring slot for its units.
//
// Reduction.  Consumer warps take the CTA's units round-robin; each unit
// leaves one partial per row in shared memory, and after a pass of units the
// CTA adds each row's partials in superblock order (deterministic).
//
// Arithmetic: 32-bit fixed-point activation digit planes and exact integer
// dp4a block sums, scales applied in fp32 (gemv_common.cuh).
#pragma once

#include "gemv_common.cuh"
#include "q4k_internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <q4k.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

namespace q4k {
namespace seq {


constexpr int kConsumerWarps = 15;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;          // + one producer warp
constexpr int kRB = 32;                            // rows per block (one per lane)
constexpr int kUnitSB = 2;                         // superblocks per unit
constexpr int kUnitBytes = kUnitSB * kRB * kBlockBytes;   // one ring slot (Q4_K units)
// Q6_K units (GPU layout): 32 rows x 2 superblocks of 208 bytes, then the
// rows' d values (an aligned group of 8 per row); a launch that holds a
// Q6_K job uses slots of this size for all its units
constexpr int kQ6UnitQuant = kUnitSB * kRB * gemv::kQ6Blk;
constexpr int kQ6UnitBytes = kQ6UnitQuant + kRB * 16;
constexpr int kLaunchQ6 = 48;                      // Q6_K jobs per launch (their d maps in the parameters)
constexpr int kFmtQ4K = 0, kFmtQ6K = 1;
static_assert(kQ6UnitQuant % 128 == 0 && kQ6UnitBytes % 128 == 0, "tensor-copy destinations 128-byte aligned");
constexpr int kMaxRing = 24;
constexpr int kLaunchJobs = 96;                    // jobs per launch (tensor maps in the parameters)
constexpr size_t kSyncBytes = 256;

struct SeqJob {
  const float* res;
  float* y;
  int rows;
  int rb_base;      // first row block of the job within its segment
  int dmap;         // Q6_K: index of the d-value map, else -1
};

struct SeqSeg {
  const float* x;
  long long unit_base;   // first unit of the segment within its epoch
  int job_begin, job_end;
  int nb;                // superblocks per row
  int nu;                // units per row block: ceil(nb / kUnitSB)
  int n_rb;              // row blocks of the segment
  int fmt;               // weight format of its jobs (kFmtQ4K, kFmtQ6K)
};

struct SeqEpoch {
  long long units;       // units of all its segments
  int seg_begin, seg_end;
  int ctas;              // CTAs sharing its units (<= grid)
  int aligned;           // CTA ranges start on row-block boundaries (no shared row blocks)
};

struct SeqParams {
  CUtensorMap map[kLaunchJobs];   // one per job: box of 144 (Q6_K: 208) bytes x 32 rows x 2 superblocks
  CUtensorMap dmap[kLaunchQ6];    // Q6_K jobs' d values: box of 8 x 32 rows
  SeqJob job[kLaunchJobs];
  SeqSeg seg[kLaunchJobs];
  SeqEpoch epoch[kLaunchJobs];
  int n_epoch;
  int ring;
  int slot_bytes;     // kUnitBytes, or kQ6UnitBytes when the launch holds a Q6_K job
  int nb_max;
  int part_floats;
  unsigned* sync;     // [0] segment arrivals, [1] CTAs exited, [2] abort
  unsigned* tickets;  // [2][grid]: pieces of a split row block stored (epoch parity)
  float* pieces;      // [2][grid][2][kRB * B]: a CTA's first / last row block
  int* err;
};

// kernel parameters are limited to 32764 bytes
static_assert(sizeof(SeqParams) <= 32000, "too many jobs per launch for the kernel parameter space");

struct SeqLayout {
  size_t xs, xss, part, carry, flags, ring, bars, total;
};

__host__ __device__ inline SeqLayout seq_layout(int B, int nb_max, int part_floats, int ring, int slot_bytes) {
  SeqLayout L;
  L.xs = 0;
  L.xss = L.xs + gemv::xs_bytes(B, nb_max);
  L.part = L.xss + gemv::xss_bytes(B, nb_max);
  L.carry = L.part + sizeof(float) * (size_t)part_floats;
  L.flags = L.carry + sizeof(float) * 2 * kRB * (size_t)B;
  L.ring = (L.flags + 16 + 127) & ~size_t(127);
  L.bars = L.ring + (size_t)ring * slot_bytes;
  L.total = L.bars + sizeof(uint64_t) * 2 * ring + 16 + 1024;   // + issue counter, + base alignment slack
  return L;
}

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_acq_rel_add_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void record_failure(const SeqParams& P) {
  atomicOr(P.err, 2);
  atomicExch(P.sync + 2, 1u);
}

// Bounded wait until `target` segment arrivals have been counted.
static __device__ __noinline__ bool grid_wait(const unsigned* counter, unsigned target) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(counter) < target) {
    __nanosleep(32);
    if (clock64() - t0 > tc::kTimeoutCycles) return false;
  }
  return true;
}

// The segment of epoch E that holds epoch unit u (binary search: a CTA far
// into a long epoch would otherwise walk dozens of segments, each a load
// from the kernel's parameter space, before its first copy).
__device__ __forceinline__ int seg_of(const SeqParams& P, const SeqEpoch& E, long long u) {
  int lo = E.seg_begin, hi = E.seg_end - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.seg[mid].unit_base <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// First unit of CTA c's range in epoch E (c = ctas gives the end): an equal
// share, or, in an aligned epoch, that share moved back to the start of its
// row block (then no row block is shared and nothing has to be combined;
// some CTAs may get no units).
__device__ __forceinline__ long long range_begin(const SeqParams& P, const SeqEpoch& E, int c) {
  const long long u = (long long)c * E.units / E.ctas;
  if (!E.aligned || c >= E.ctas) return u;
  const SeqSeg& S = P.seg[seg_of(P, E, u)];
  return S.unit_base + (u - S.unit_base) / S.nu * S.nu;
}

// The CTA whose range holds epoch unit u (in epochs that are not aligned;
// only those share row blocks).
__device__ __forceinline__ int owner_of(const SeqEpoch& E, long long u) {
  return (int)(((u + 1) * E.ctas + E.units - 1) / E.units - 1);
}

// The job of segment S that holds row block rb (binary search).
__device__ __forceinline__ int job_of(const SeqParams& P, const SeqSeg& S, long long rb) {
  int lo = S.job_begin, hi = S.job_end - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.job[mid].rb_base <= rb) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Piece held by CTA c of the row block whose units are epoch units
// [f, f + nu): side 0 if it is c's first row block, else side 1.
__device__ __forceinline__ float* piece_of(const SeqParams& P, const SeqEpoch& E, int slot, int grid, int c,
                                           long long f, int nu, int B) {
  const long long u0 = (long long)c * E.units / E.ctas;
  const int side = (u0 >= f && u0 < f + nu) ? 0 : 1;
  return P.pieces + (((size_t)slot * grid + c) * 2 + side) * (size_t)(kRB * B);
}

// Consumer warps over slots [ps, pe) of a run of one segment's units: slot s
// is segment unit u0 + s and stage J + s.  Each unit leaves 32 partial row
// sums (its two superblocks added in order) in part[s - ps][row][b].
template <int B, int FMT>
__device__ __forceinline__ void consume_pass(const SeqParams& P, const uint8_t* ring_base, int slot_bytes,
                                             uint64_t* full, uint64_t* empty, volatile int* issued, int ring,
                                             int J, int ps, int pe, long long u0, int nb, int nu,
                                             const gemv::XView& xv, float* part, bool& ok, int warp, int lane) {
  for (int s = ps + warp; s < pe; s += kConsumerWarps) {
    const int j = J + s;
    const int slot = j % ring;
    const uint32_t parity = (uint32_t)((j / ring) & 1);
    // a warp that skips stages must see stage j issued before it waits on
    // its parity (the copy of stage j - ring may still be in flight)
    if (ok && *issued <= j && !gemv::wait_issued(issued, j)) {
      ok = false;
      if (lane == 0) record_failure(P);
    }
    if (ok && !tc::mbar_wait_spin(&full[slot], parity)) {
      ok = false;
      if (lane == 0) record_failure(P);
    }
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    if (ok) {
      const int sb = (int)((u0 + s) % nu) * kUnitSB;
      const uint8_t* slot_p = ring_base + (size_t)slot * slot_bytes;
      if constexpr (FMT == kFmtQ6K) {
        // [superblock][row][208], then d as [row][8] for the aligned group holding sb
        const uint8_t* p = slot_p + lane * gemv::kQ6Blk;
        const __half* dv = reinterpret_cast<const __half*>(slot_p + kQ6UnitQuant) + lane * 8 + (sb & 7);
        gemv::superblock_dot_q6<B, 4, true>(p, __half2float(dv[0]), xv, sb, 0, acc);
        if (sb + 1 < nb) {
          float acc2[B];
          gemv::superblock_dot_q6<B, 4, true>(p + kRB * gemv::kQ6Blk, __half2float(dv[1]), xv, sb + 1, 0, acc2);
#pragma unroll
          for (int b = 0; b < B; ++b) acc[b] += acc2[b];
        }
      } else {
        const uint8_t* p = slot_p + lane * kBlockBytes;
        gemv::superblock_dot<B, 4, true>(p, xv, sb, 0, acc);
        if (sb + 1 < nb) {
          float acc2[B];
          gemv::superblock_dot<B, 4, true>(p + kRB * kBlockBytes, xv, sb + 1, 0, acc2);
#pragma unroll
          for (int b = 0; b < B; ++b) acc[b] += acc2[b];
        }
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[slot]);
#pragma unroll
    for (int b = 0; b < B; ++b) part[((size_t)(s - ps) * kRB + lane) * B + b] = acc[b];
  }
}

// Row sums of the segment units [ua, ub) of this pass, where [u0, u1) is the
// CTA's part of the segment, in superblock order.  A row block whose part
// continues into the next pass leaves its sum in carry_out; one that began
// in the previous pass starts from carry_in.  A row block finished here is
// stored to y, or, if the CTA's range cuts it, to this CTA's piece of it.
template <int B>
__device__ __forceinline__ void reduce_pass(const SeqParams& P, const SeqSeg& S, const SeqEpoch& E, int slot,
                                            long long u0, long long u1, long long ua, long long ub,
                                            const float* part, const float* carry_in, float* carry_out, int c,
                                            int grid, int tid) {
  const int nu = S.nu;   // units per row block
  const long long rb_lo = ua / nu, rb_hi = (ub - 1) / nu;
  const int n_rbp = (int)(rb_hi - rb_lo + 1);
  constexpr int per = kRB * B;
  for (int i = tid; i < n_rbp * per; i += kConsumers) {
    const int k = i / per, rem = i - k * per, r = rem / B, b = rem - r * B;
    const long long rb = rb_lo + k;
    const long long first = rb * nu, last = first + nu;
    const long long a = first > ua ? first : ua, e = last < ub ? last : ub;
    float v = ((first > u0 ? first : u0) < ua) ? carry_in[rem] : 0.0f;
    for (long long uu = a; uu < e; ++uu) v += part[((uu - ua) * kRB + r) * B + b];
    if ((last < u1 ? last : u1) > ub) {
      carry_out[rem] = v;
      continue;
    }
    if (first < u0 || last > u1) {
      piece_of(P, E, slot, grid, c, S.unit_base + first, nu, B)[rem] = v;
      continue;
    }
    const SeqJob& Jb = P.job[job_of(P, S, rb)];
    const long long row = (rb - Jb.rb_base) * kRB + r;
    if (row >= Jb.rows) continue;
    if (Jb.res) v += __ldcg(Jb.res + (size_t)b * Jb.rows + row);
    Jb.y[(size_t)b * Jb.rows + row] = v;
  }
}

// Q6: the launch holds Q6_K jobs (lists of Q4_K jobs only run the variant
// without the Q6_K path, which keeps its registers and code for the Q4_K one)
template <int B, bool Q6>
__global__ void __launch_bounds__(kThreads, 1) gemv_seq_kernel(const __grid_constant__ SeqParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int ring = P.ring;
  const int slot_bytes = Q6 ? P.slot_bytes : kUnitBytes;
  const SeqLayout L = seq_layout(B, P.nb_max, P.part_floats, ring, slot_bytes);
  uint8_t* xs = smem + L.xs;
  float2* xss = reinterpret_cast<float2*>(smem + L.xss);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* carry = reinterpret_cast<float*>(smem + L.carry);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  uint8_t* ring_base = smem + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + ring;
  volatile int* issued = reinterpret_cast<volatile int*>(empty + ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, grid = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < ring; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    *issued = 0;
    flags[0] = flags[1] = flags[2] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0, slot = 0;
      uint32_t phase = 0;
      bool pok = true;
      for (int ei = 0; ei < P.n_epoch && pok; ++ei) {
        const SeqEpoch& E = P.epoch[ei];
        if (c >= E.ctas) continue;
        const long long e1 = range_begin(P, E, c + 1);
        long long u = range_begin(P, E, c);
        int si = seg_of(P, E, u);
        while (u < e1 && pok) {
          const SeqSeg& S = P.seg[si];
          const int nu = S.nu;
          const long long su1 = S.unit_base + (long long)S.n_rb * nu;
          const long long end = e1 < su1 ? e1 : su1;
          long long rb = (u - S.unit_base) / nu;
          int up = (int)(u - S.unit_base - rb * nu);
          int jb = job_of(P, S, rb);
          for (; u < end; ++u) {
            if (!tc::mbar_wait_spin(&empty[slot], phase ^ 1)) {
              record_failure(P);
              pok = false;
              break;
            }
            uint8_t* dst = ring_base + (size_t)slot * slot_bytes;
            const int row = (int)(rb - P.job[jb].rb_base) * kRB;
            if (Q6 && S.fmt == kFmtQ6K) {
              tc::mbar_arrive_expect_tx(&full[slot], kQ6UnitBytes);
              tc::tma_load_3d(dst, &P.map[jb], 0, row, up * kUnitSB, &full[slot]);
              tc::tma_load_2d(dst + kQ6UnitQuant, &P.dmap[P.job[jb].dmap], (up * kUnitSB) & ~7, row, &full[slot]);
            } else {
              tc::mbar_arrive_expect_tx(&full[slot], kUnitBytes);
              tc::tma_load_3d(dst, &P.map[jb], 0, row, up * kUnitSB, &full[slot]);
            }
            __threadfence_block();
            *issued = ++j;
            if (++slot == ring) {
              slot = 0;
              phase ^= 1;
            }
            if (++up == nu) {
              up = 0;
              ++rb;
              if (jb + 1 < S.job_end && rb >= P.job[jb + 1].rb_base) ++jb;
            }
          }
          ++si;
        }
      }
      // every copy issued has landed before the CTA exits, even if consumers
      // gave up a wait and left early (bounded as well)
      for (int k = max(0, j - ring); k < j; ++k)
        if (!tc::mbar_wait_sleep(&full[k % ring], (uint32_t)((k / ring) & 1))) record_failure(P);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  bool ok = true;
  const float* staged_x = nullptr;
  int staged_nb = -1;
  int J = 0;          // this CTA's stages so far (ring order)
  int pass_no = 0;
  constexpr int per = kRB * B;
  for (int ei = 0; ei < P.n_epoch; ++ei) {
    const SeqEpoch& E = P.epoch[ei];
    const int slot = ei & 1;
    long long e0 = 0, e1 = 0;
    if (c < E.ctas) {
      e0 = range_begin(P, E, c);
      e1 = range_begin(P, E, c + 1);
    }
    if (ei > 0) {
      // activations may be outputs of earlier jobs: wait for all of them
      if (tid == 0 && ok && !grid_wait(P.sync, (unsigned)ei * (unsigned)grid)) {
        record_failure(P);
        flags[2] = 1;
      }
      named_sync_consumers();
      ok = ok && !flags[2];
      staged_x = nullptr;
    }
    for (long long u = e0; u < e1;) {
      const int si = seg_of(P, E, u);
      const SeqSeg& S = P.seg[si];
      const int nb = S.nb, nu = S.nu;
      const long long su1 = S.unit_base + (long long)S.n_rb * nu;
      const long long u0 = u - S.unit_base, u1 = (e1 < su1 ? e1 : su1) - S.unit_base;   // segment units
      const int n_units = (int)(u1 - u0);
      if (S.x != staged_x || nb != staged_nb) {
        gemv::stage_x<B, kConsumers, true>(S.x, nb, xs, xss, tid);
        staged_x = S.x;
        staged_nb = nb;
        named_sync_consumers();
      }
      const int pu = P.part_floats / per;   // units per pass
      for (int ps = 0; ps < n_units; ps += pu, ++pass_no) {
        const int pe = min(ps + pu, n_units);
        bool q6_seg = false;
        if constexpr (Q6) {
          if (S.fmt == kFmtQ6K) {
            q6_seg = true;
            consume_pass<B, kFmtQ6K>(P, ring_base, slot_bytes, full, empty, issued, ring, J, ps, pe, u0, nb, nu,
                                     gemv::make_view(xs, xss, S.x, B, nb), part, ok, warp, lane);
          }
        }
        if (!q6_seg)
          consume_pass<B, kFmtQ4K>(P, ring_base, slot_bytes, full, empty, issued, ring, J, ps, pe, u0, nb, nu,
                                   gemv::make_view(xs, xss, S.x, B, nb), part, ok, warp, lane);
        if (!ok) flags[2] = 1;
        named_sync_consumers();
        ok = ok && !flags[2];
        if (ok)
          reduce_pass<B>(P, S, E, slot, u0, u1, u0 + ps, u0 + pe, part, carry + (pass_no & 1) * per,
                         carry + ((pass_no + 1) & 1) * per, c, grid, tid);
        named_sync_consumers();
      }
      J += n_units;
      u += n_units;
    }
    if (e1 > e0 && ok) {
      // row blocks cut by this CTA's range: the last holder adds the pieces
      const int s_first = seg_of(P, E, e0), s_last = seg_of(P, E, e1 - 1);
      const SeqSeg& Sf = P.seg[s_first];
      const SeqSeg& Sl = P.seg[s_last];
      const long long f_first = Sf.unit_base + (e0 - Sf.unit_base) / Sf.nu * Sf.nu;   // first unit of the row block
      const long long f_last = Sl.unit_base + (e1 - 1 - Sl.unit_base) / Sl.nu * Sl.nu;
      const bool split_first = f_first < e0 || f_first + Sf.nu > e1;
      const bool split_last = f_last != f_first && f_last + Sl.nu > e1;
      if (split_first || split_last) {
        if (tid < 2) {
          const bool mine = tid == 0 ? split_first : split_last;
          int fl = 0;
          if (mine) {
            const long long f = tid == 0 ? f_first : f_last;
            const int nbs = tid == 0 ? Sf.nu : Sl.nu;
            const int c0 = owner_of(E, f), c1 = owner_of(E, f + nbs - 1);
            unsigned* t = P.tickets + (size_t)slot * grid + c1;
            if (atom_acq_rel_add_gpu(t, 1u) == (unsigned)(c1 - c0)) {
              fl = 1;
              atomicExch(t, 0u);
            }
          }
          flags[tid] = fl;
        }
        named_sync_consumers();
        const int fl = flags[0] | (flags[1] << 1);
        for (int i = tid; i < 2 * per; i += kConsumers) {
          const int side = i / per, rem = i - side * per;
          if (!(fl & (1 << side))) continue;
          const SeqSeg& S = side == 0 ? Sf : Sl;
          const long long f = side == 0 ? f_first : f_last;
          const long long rb = (f - S.unit_base) / S.nu;
          const int r = rem / B, b = rem - r * B;
          const SeqJob& Jb = P.job[job_of(P, S, rb)];
          const long long row = (rb - Jb.rb_base) * kRB + r;
          if (row >= Jb.rows) continue;
          const int c0 = owner_of(E, f), c1 = owner_of(E, f + S.nu - 1);
          float v = 0.0f;
          for (int cc = c0; cc <= c1; ++cc) v += __ldcg(piece_of(P, E, slot, grid, cc, f, S.nu, B) + rem);
          if (Jb.res) v += __ldcg(Jb.res + (size_t)b * Jb.rows + row);
          Jb.y[(size_t)b * Jb.rows + row] = v;
        }
      }
    }
    // every output of this CTA for the epoch is stored: count the arrival
    named_sync_consumers();
    if (tid == 0) red_release_add_gpu(P.sync, 1u);
  }

  // the last CTA out resets the workspace for the next launch
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.sync + 1, 1u) == (unsigned)grid - 1) {
      if (atomicAdd(P.sync + 2, 0u) != 0u) {
        for (int i = 0; i < 2 * grid; ++i) P.tickets[i] = 0u;
        P.sync[2] = 0u;
      }
      atomicExch(P.sync, 0u);
      atomicExch(P.sync + 1, 0u);
      __threadfence();
    }
  }
}

// Shared-memory opt-in and launch of one kernel variant (Q6: the launch holds
// Q6_K jobs).  Explicitly instantiated in gemv_seq_q4.cu (Q6 = false) and
// gemv_seq_q6a.cu / q6b / q6c (Q6 = true, batch 1-4 / 5-6 / 7-8), so
// that no translation unit takes long to compile.
template <int B, bool Q6>
cudaError_t set_smem(int max_smem) {
  return cudaFuncSetAttribute(gemv_seq_kernel<B, Q6>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

template <int B, bool Q6>
cudaError_t launch(const SeqParams& P, unsigned grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // every CTA must be resident at once: CTAs wait for one another's arrivals
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_seq_kernel<B, Q6>, P);
}

#define Q4K_SEQ_VARIANTS_1_4(X, Q6) X(1, Q6) X(2, Q6) X(3, Q6) X(4, Q6)
#define Q4K_SEQ_VARIANTS_5_6(X, Q6) X(5, Q6) X(6, Q6)
#define Q4K_SEQ_VARIANTS_7_8(X, Q6) X(7, Q6) X(8, Q6)
#define Q4K_SEQ_VARIANTS(X, Q6) Q4K_SEQ_VARIANTS_1_4(X, Q6) Q4K_SEQ_VARIANTS_5_6(X, Q6) Q4K_SEQ_VARIANTS_7_8(X, Q6)
#define Q4K_SEQ_DECLARE(B, Q6)                                     \
  extern template cudaError_t set_smem<B, Q6>(int);                \
  extern template cudaError_t launch<B, Q6>(const SeqParams&, unsigned, size_t, cudaStream_t);
#define Q4K_SEQ_DEFINE(B, Q6)                                      \
  template cudaError_t set_smem<B, Q6>(int);                       \
  template cudaError_t launch<B, Q6>(const SeqParams&, unsigned, size_t, cudaStream_t);

}  // namespace seq
}  // namespace q4k
