// q4k_gemv_seq: an ordered list of decode GEMV jobs y = W x (+ residual) over
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
namespace {

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
__device__ __noinline__ bool grid_wait(const unsigned* counter, unsigned target) {
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
__device__ __forceinline__ void consume_pass(const SeqParams& P, const uint8_t* ring_base, uint64_t* full,
                                             uint64_t* empty, volatile int* issued, int ring, int J, int ps,
                                             int pe, long long u0, int nb, int nu, const gemv::XView& xv,
                                             float* part, bool& ok, int warp, int lane) {
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
      const uint8_t* slot_p = ring_base + (size_t)slot * P.slot_bytes;
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

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_seq_kernel(const __grid_constant__ SeqParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int ring = P.ring;
  const SeqLayout L = seq_layout(B, P.nb_max, P.part_floats, ring, P.slot_bytes);
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
            uint8_t* dst = ring_base + (size_t)slot * P.slot_bytes;
            const int row = (int)(rb - P.job[jb].rb_base) * kRB;
            if (S.fmt == kFmtQ6K) {
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
        if (S.fmt == kFmtQ6K)
          consume_pass<B, kFmtQ6K>(P, ring_base, full, empty, issued, ring, J, ps, pe, u0, nb, nu,
                                   gemv::make_view(xs, xss, S.x, B, nb), part, ok, warp, lane);
        else
          consume_pass<B, kFmtQ4K>(P, ring_base, full, empty, issued, ring, J, ps, pe, u0, nb, nu,
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

struct SeqPlan {
  int n_seg, n_epoch, nb_max, ring, part_floats, grid;
  size_t smem, ws_bytes, tickets_off, pieces_off;
};

// Whether an epoch's CTA ranges should start on row-block boundaries.  The
// equal shares cost the largest share plus, when a boundary falls inside a
// row block, the combine of shared row blocks at the epoch's end (a ticket
// and a gather through L2: measured at 2-3 us, about kCombineUnits units of
// streaming); the aligned ranges cost their largest range.  The smaller
// estimate wins: small epochs (a decode layer's o or down projection in
// engine order) go aligned, large ones keep equal shares.
constexpr long long kCombineUnits = 12;

bool choose_aligned(const SeqEpoch& E, const SeqSeg* seg) {
  auto seg_at = [&](long long u) {
    int s = E.seg_begin;
    while (s + 1 < E.seg_end && u >= seg[s + 1].unit_base) ++s;
    return s;
  };
  auto snapped = [&](int c) -> long long {
    const long long u = (long long)c * E.units / E.ctas;
    if (c >= E.ctas) return u;
    const SeqSeg& S = seg[seg_at(u)];
    return S.unit_base + (u - S.unit_base) / S.nu * S.nu;
  };
  long long equal_max = 0, aligned_max = 0;
  bool shared = false;
  for (int c = 0; c < E.ctas; ++c) {
    const long long u0 = (long long)c * E.units / E.ctas, u1 = (long long)(c + 1) * E.units / E.ctas;
    equal_max = std::max(equal_max, u1 - u0);
    if (c > 0 && snapped(c) != u0) shared = true;
    aligned_max = std::max(aligned_max, snapped(c + 1) - snapped(c));
  }
  return aligned_max < equal_max + (shared ? kCombineUnits : 0);
}

// Segments, epochs, row blocks and CTA shares of one launch's jobs (at most
// kLaunchJobs).  Fills P (if not null) and the plan; returns a status.
int plan_launch(const q4k_gemv_job* jobs, int n_jobs, int B, const DeviceInfo& info, SeqParams* P,
                SeqPlan* plan) {
  SeqPlan p{};
  p.grid = info.sm_count;
  int n_seg = 0, n_job = 0, n_epoch = 0;
  SeqSeg tseg[kLaunchJobs];
  SeqJob tjob[kLaunchJobs];
  SeqEpoch tep[kLaunchJobs];
  const void* tw[kLaunchJobs];
  int64_t tcols[kLaunchJobs];
  int tfmt[kLaunchJobs];
  int n_q6 = 0;
  bool pending_wait = false;
  const float* cur_x = nullptr;
  int cur_nb = -1, cur_fmt = -1;
  for (int i = 0; i < n_jobs; ++i) {
    const q4k_gemv_job& q = jobs[i];
    pending_wait = pending_wait || q.wait != 0;
    if (q.rows == 0) continue;
    const int nb = (int)(q.cols / kQK);
    const int fmt = q.format == 1 ? kFmtQ6K : kFmtQ4K;
    // a segment holds one weight format (same x across a format change:
    // the next segment does not stage x again)
    if (n_seg == 0 || pending_wait || q.x != cur_x || nb != cur_nb || fmt != cur_fmt) {
      if (n_seg > 0) tseg[n_seg - 1].job_end = n_job;
      if (n_seg == 0 || pending_wait) {
        if (n_epoch > 0) tep[n_epoch - 1].seg_end = n_seg;
        SeqEpoch e{};
        e.seg_begin = n_seg;
        tep[n_epoch++] = e;
      }
      SeqSeg sg{};
      sg.x = q.x;
      sg.job_begin = n_job;
      sg.nb = nb;
      sg.fmt = fmt;
      tseg[n_seg++] = sg;
      cur_x = q.x;
      cur_nb = nb;
      cur_fmt = fmt;
      pending_wait = false;
    }
    SeqJob jb{};
    jb.res = q.residual;
    jb.y = q.y;
    jb.rows = (int)q.rows;
    jb.dmap = -1;
    if (fmt == kFmtQ6K) {
      if (n_q6 == kLaunchQ6) return Q4K_ERR_UNSUPPORTED;   // (the chunking keeps launches below this)
      jb.dmap = n_q6++;
    }
    tw[n_job] = q.w;
    tcols[n_job] = q.cols;
    tfmt[n_job] = fmt;
    tjob[n_job++] = jb;
  }
  if (n_seg > 0) tseg[n_seg - 1].job_end = n_job;
  if (n_epoch > 0) tep[n_epoch - 1].seg_end = n_seg;
  p.n_seg = n_seg;
  p.n_epoch = n_epoch;
  p.nb_max = 1;
  for (int e = 0; e < n_epoch; ++e) {
    SeqEpoch& E = tep[e];
    int64_t units = 0;
    for (int s = E.seg_begin; s < E.seg_end; ++s) {
      SeqSeg& S = tseg[s];
      int64_t n_rb = 0;
      for (int j = S.job_begin; j < S.job_end; ++j) {
        tjob[j].rb_base = (int)n_rb;
        n_rb += (tjob[j].rows + kRB - 1) / kRB;
      }
      S.n_rb = (int)n_rb;
      S.nu = (S.nb + kUnitSB - 1) / kUnitSB;
      S.unit_base = units;
      units += n_rb * S.nu;
      p.nb_max = std::max(p.nb_max, S.nb);
    }
    if (units / p.grid > (int64_t(1) << 30)) return Q4K_ERR_UNSUPPORTED;
    E.units = units;
    E.ctas = (int)std::min<int64_t>(p.grid, units);
    E.aligned = choose_aligned(E, tseg) ? 1 : 0;
  }
  // shared memory: activations, partial sums, then the deepest ring that fits
  p.part_floats = 16 * kRB * B * (B == 1 ? 16 : (B == 2 ? 8 : (B <= 4 ? 2 : 1)));
  p.ring = 0;
  const int slot_bytes = n_q6 > 0 ? kQ6UnitBytes : kUnitBytes;
  for (int ring = kMaxRing; ring >= 4; --ring) {
    const size_t total = seq_layout(B, p.nb_max, p.part_floats, ring, slot_bytes).total;
    if (total <= (size_t)info.max_smem_optin) {
      p.ring = ring;
      p.smem = total;
      break;
    }
  }
  if (p.ring == 0) return Q4K_ERR_UNSUPPORTED;
  // workspace: counters, then per epoch parity one ticket and two pieces per CTA
  const size_t tickets_bytes = ((sizeof(unsigned) * 2 * (size_t)p.grid) + 255) & ~size_t(255);
  p.tickets_off = kSyncBytes;
  p.pieces_off = kSyncBytes + tickets_bytes;
  p.ws_bytes = p.pieces_off + sizeof(float) * 2 * (size_t)p.grid * 2 * kRB * B;
  if (P) {
    for (int j = 0; j < n_job; ++j) {
      // box: a superblock's 144 (Q6_K: 208) bytes x 32 rows x 2 superblocks;
      // rows and superblocks past the matrix read as zeros
      const uint64_t nbj = (uint64_t)(tcols[j] / kQK);
      const bool q6 = tfmt[j] == kFmtQ6K;
      const uint64_t blk = q6 ? (uint64_t)gemv::kQ6Blk : (uint64_t)kBlockBytes;
      const uint64_t row_bytes = q6 ? (uint64_t)q6k_gpu_row_bytes((int64_t)nbj) : nbj * kBlockBytes;
      const uint64_t dims[3] = {blk, (uint64_t)tjob[j].rows, nbj};
      const uint64_t strides[2] = {row_bytes, blk};
      const uint32_t box[3] = {(uint32_t)blk, (uint32_t)kRB, (uint32_t)kUnitSB};
      if (!encode_tmap_u8_3d(&P->map[j], tw[j], dims, strides, box)) return Q4K_ERR_CUDA;
      // Q6_K: the rows' d values after their superblocks, 8 x 32 rows a box
      if (q6 && !encode_tmap_2d(&P->dmap[tjob[j].dmap], CU_TENSOR_MAP_DATA_TYPE_UINT16,
                                static_cast<const uint8_t*>(tw[j]) + nbj * blk, nbj, (uint64_t)tjob[j].rows,
                                row_bytes, 8, (uint32_t)kRB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q4K_ERR_CUDA;
    }
    std::memcpy(P->seg, tseg, sizeof(SeqSeg) * n_seg);
    std::memcpy(P->job, tjob, sizeof(SeqJob) * n_job);
    std::memcpy(P->epoch, tep, sizeof(SeqEpoch) * n_epoch);
    P->n_epoch = n_epoch;
    P->ring = p.ring;
    P->slot_bytes = slot_bytes;
    P->nb_max = p.nb_max;
    P->part_floats = p.part_floats;
  }
  *plan = p;
  return Q4K_OK;
}

// Set once per device and batch: the kernel may use the opt-in shared memory.
template <int B>
cudaError_t allow_smem(int dev, const DeviceInfo& info) {
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if (limit < info.max_smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_seq_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin);
    if (e != cudaSuccess) return e;
    limit = info.max_smem_optin;
  }
  return cudaSuccess;
}

cudaError_t allow_smem_batch(int batch, int dev, const DeviceInfo& info) {
  switch (batch) {
    case 1: return allow_smem<1>(dev, info);
    case 2: return allow_smem<2>(dev, info);
    case 3: return allow_smem<3>(dev, info);
    case 4: return allow_smem<4>(dev, info);
    case 5: return allow_smem<5>(dev, info);
    case 6: return allow_smem<6>(dev, info);
    case 7: return allow_smem<7>(dev, info);
    case 8: return allow_smem<8>(dev, info);
    default: return cudaErrorNotSupported;
  }
}

template <int B>
cudaError_t launch_seq_b(const SeqParams& P, const SeqPlan& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  // every CTA must be resident at once: CTAs wait for one another's arrivals
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_seq_kernel<B>, P);
}

cudaError_t launch_seq_batch(const SeqParams& P, const SeqPlan& p, int batch, cudaStream_t s) {
  switch (batch) {
    case 1: return launch_seq_b<1>(P, p, s);
    case 2: return launch_seq_b<2>(P, p, s);
    case 3: return launch_seq_b<3>(P, p, s);
    case 4: return launch_seq_b<4>(P, p, s);
    case 5: return launch_seq_b<5>(P, p, s);
    case 6: return launch_seq_b<6>(P, p, s);
    case 7: return launch_seq_b<7>(P, p, s);
    case 8: return launch_seq_b<8>(P, p, s);
    default: return cudaErrorNotSupported;
  }
}

// Launches of a job list: consecutive chunks of at most kLaunchJobs jobs
// (stream order between launches is a full dependency), each holding at most
// kLaunchQ6 Q6_K jobs with work
int next_chunk(const q4k_gemv_job* jobs, int i0, int n_jobs) {
  int i = i0, q6 = 0;
  while (i < n_jobs && i - i0 < kLaunchJobs) {
    if (jobs[i].format == 1 && jobs[i].rows > 0) {
      if (q6 == kLaunchQ6) break;
      ++q6;
    }
    ++i;
  }
  return i;
}
// an upper bound on the launches of any list of n_jobs jobs (plan buffers)
int n_launches(int n_jobs) { return n_jobs <= 0 ? 1 : (n_jobs + kLaunchQ6 - 1) / kLaunchQ6; }

// A prepared job list in caller-owned host memory: a header, then one
// (kernel parameters, launch shape) pair per launch.
constexpr uint64_t kPlanMagic = 0x71346b5365715031ull;   // "q4kSeqP1"

struct SeqLaunch {
  SeqParams P;       // first: the tensor maps need 64-byte alignment
  SeqPlan plan;
  int active;        // 0: the chunk holds no work (every job has 0 rows)
};

struct alignas(64) PlanHeader {
  uint64_t magic;
  int n_launch, batch, dev;
  size_t ws_need;     // workspace bytes the launches need
  size_t counters;    // leading workspace bytes that must start at zero
  const void* ws;     // bound workspace
};

size_t plan_bytes_for(int n_jobs) {
  return sizeof(PlanHeader) + sizeof(SeqLaunch) * (size_t)n_launches(n_jobs);
}

// Plan every launch of a job list into `buf`: segments, epochs, CTA shares,
// tensor maps, the workspace it needs.  Enqueues nothing.  With `ws` null
// the workspace is bound later (bind_workspace).
int build_plan(const q4k_gemv_job* jobs, int n_jobs, int batch, void* buf, size_t bytes, cudaError_t* ce) {
  *ce = cudaSuccess;
  if (bytes < plan_bytes_for(n_jobs)) return Q4K_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(buf) & 63u) != 0) return Q4K_ERR_ALIGNMENT;
  int dev = 0;
  if ((*ce = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
  if (dev < 0 || dev >= 64) return Q4K_ERR_UNSUPPORTED;
  const DeviceInfo& info = device_info(dev);
  int* err = device_error_word();
  if (!err) {
    *ce = cudaGetLastError();
    return Q4K_ERR_CUDA;
  }
  PlanHeader* h = static_cast<PlanHeader*>(buf);
  SeqLaunch* L = reinterpret_cast<SeqLaunch*>(static_cast<uint8_t*>(buf) + sizeof(PlanHeader));
  h->magic = 0;
  size_t need = kSyncBytes;
  int k = 0;
  for (int i0 = 0; i0 < n_jobs || k == 0; i0 = next_chunk(jobs, i0, n_jobs), ++k) {
    SeqLaunch& l = L[k];
    std::memset(&l.P, 0, sizeof(l.P));
    const int st = plan_launch(jobs + i0, next_chunk(jobs, i0, n_jobs) - i0, batch, info, &l.P, &l.plan);
    if (st == Q4K_ERR_CUDA) *ce = cudaErrorInvalidValue;   // a tensor map the driver refused
    if (st != Q4K_OK) return st;
    l.active = l.plan.n_epoch > 0;
    l.P.err = err;
    need = std::max(need, l.plan.ws_bytes);
    if (n_jobs == 0) {
      ++k;
      break;
    }
  }
  if ((*ce = allow_smem_batch(batch, dev, info)) != cudaSuccess) return Q4K_ERR_CUDA;
  h->n_launch = k;
  h->batch = batch;
  h->dev = dev;
  h->ws_need = need;
  h->counters = kSyncBytes + (((sizeof(unsigned) * 2 * (size_t)info.sm_count) + 255) & ~size_t(255));
  h->ws = nullptr;
  h->magic = kPlanMagic;
  return Q4K_OK;
}

int bind_workspace(void* buf, void* ws, size_t ws_bytes) {
  PlanHeader* h = static_cast<PlanHeader*>(buf);
  if (ws_bytes < h->ws_need) return Q4K_ERR_INVALID_ARG;
  SeqLaunch* L = reinterpret_cast<SeqLaunch*>(static_cast<uint8_t*>(buf) + sizeof(PlanHeader));
  uint8_t* w = static_cast<uint8_t*>(ws);
  for (int k = 0; k < h->n_launch; ++k) {
    L[k].P.sync = reinterpret_cast<unsigned*>(w);
    L[k].P.tickets = reinterpret_cast<unsigned*>(w + L[k].plan.tickets_off);
    L[k].P.pieces = reinterpret_cast<float*>(w + L[k].plan.pieces_off);
  }
  h->ws = ws;
  return Q4K_OK;
}

int run_plan(const void* buf, cudaStream_t s, cudaError_t* ce) {
  *ce = cudaSuccess;
  const PlanHeader* h = static_cast<const PlanHeader*>(buf);
  if (h->magic != kPlanMagic || !h->ws) return Q4K_ERR_INVALID_ARG;
  int dev = 0;
  if ((*ce = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
  if (dev != h->dev) return Q4K_ERR_INVALID_ARG;
  const SeqLaunch* L = reinterpret_cast<const SeqLaunch*>(static_cast<const uint8_t*>(buf) + sizeof(PlanHeader));
  for (int k = 0; k < h->n_launch; ++k) {
    if (!L[k].active) continue;
    if ((*ce = launch_seq_batch(L[k].P, L[k].plan, h->batch, s)) != cudaSuccess) return Q4K_ERR_CUDA;
  }
  return Q4K_OK;
}

// Per-thread plan buffer of the one-shot entry points (a job list of the
// maximum length takes three launches).
struct alignas(64) OneShotPlan {
  // room for the most launches any list can take (n_launches(kGemvSeqMaxJobs))
  uint8_t bytes[sizeof(PlanHeader) + sizeof(SeqLaunch) * ((kGemvSeqMaxJobs + kLaunchQ6 - 1) / kLaunchQ6)];
};
OneShotPlan* one_shot_plan() {
  static thread_local OneShotPlan* p = new OneShotPlan;
  return p;
}

}  // namespace

int gemv_seq_workspace(const q4k_gemv_job* jobs, int n_jobs, int batch, size_t* bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
  const DeviceInfo& info = device_info(dev);
  size_t need = kSyncBytes;
  for (int i0 = 0; i0 < n_jobs; i0 = next_chunk(jobs, i0, n_jobs)) {
    SeqPlan p;
    const int st = plan_launch(jobs + i0, next_chunk(jobs, i0, n_jobs) - i0, batch, info, nullptr, &p);
    if (st != Q4K_OK) return st;
    need = std::max(need, p.ws_bytes);
  }
  *bytes = need;
  return Q4K_OK;
}

size_t gemv_seq_plan_bytes(int n_jobs) { return plan_bytes_for(n_jobs); }

int gemv_seq_plan(const q4k_gemv_job* jobs, int n_jobs, int batch, void* workspace, size_t workspace_bytes,
                  void* plan, size_t plan_bytes, cudaError_t* cuda_err) {
  if (batch == 0 || !workspace) {
    // nothing to launch (the caller checked that no job has work)
    *cuda_err = cudaSuccess;
    if (plan_bytes < sizeof(PlanHeader)) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(plan) & 63u) != 0) return Q4K_ERR_ALIGNMENT;
    PlanHeader* h = static_cast<PlanHeader*>(plan);
    int dev = 0;
    if ((*cuda_err = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
    h->n_launch = 0;
    h->batch = batch;
    h->dev = dev;
    h->ws_need = h->counters = 0;
    h->ws = plan;
    h->magic = kPlanMagic;
    return Q4K_OK;
  }
  const int st = build_plan(jobs, n_jobs, batch, plan, plan_bytes, cuda_err);
  if (st != Q4K_OK) return st;
  const int b = bind_workspace(plan, workspace, workspace_bytes);
  if (b != Q4K_OK) static_cast<PlanHeader*>(plan)->magic = 0;
  return b;
}

int gemv_seq_launch(const void* plan, cudaStream_t s, cudaError_t* cuda_err) { return run_plan(plan, s, cuda_err); }

int launch_gemv_seq(const q4k_gemv_job* jobs, int n_jobs, int batch, void* workspace, size_t workspace_bytes,
                    cudaStream_t s, cudaError_t* cuda_err) {
  // plan every launch before enqueuing any, so that a refused request
  // enqueues nothing
  OneShotPlan* buf = one_shot_plan();
  const int st = gemv_seq_plan(jobs, n_jobs, batch, workspace, workspace_bytes, buf->bytes, sizeof(buf->bytes),
                               cuda_err);
  if (st != Q4K_OK) return st;
  return run_plan(buf->bytes, s, cuda_err);
}

// ---------------------------------------------------------------------------
// Variant that allocates nothing: the workspace is a fixed array in this
// library's device memory instead of caller-provided memory.
namespace {
constexpr size_t kStaticScratchBytes = size_t(1) << 20;   // 1 MiB
std::mutex g_static_mutex;
void* g_static_ptr[64];
}  // namespace

// Built-in workspace of q4k_gemv_seq_static.  Every GPU that loads the
// library holds it until the process exits; all calls on a device share it.
static __device__ __align__(256) unsigned char g_seq_scratch[kStaticScratchBytes];

int launch_gemv_seq_static(const q4k_gemv_job* jobs, int n_jobs, int batch, cudaStream_t s,
                           cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  int dev = 0;
  if ((*cuda_err = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
  if (dev < 0 || dev >= 64) return Q4K_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    // host code only knows the array's device address once it asks for it,
    // with the device current; the answer is kept per device
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_seq_scratch);
      if (e != cudaSuccess) {
        *cuda_err = e;
        return Q4K_ERR_CUDA;
      }
      g_static_ptr[dev] = p;
    }
    scratch = g_static_ptr[dev];
  }
  // plan (and refuse) everything before anything is enqueued
  OneShotPlan* buf = one_shot_plan();
  const int st = build_plan(jobs, n_jobs, batch, buf->bytes, sizeof(buf->bytes), cuda_err);
  if (st != Q4K_OK) return st;
  const PlanHeader* h = reinterpret_cast<const PlanHeader*>(buf->bytes);
  if (h->ws_need > kStaticScratchBytes) return Q4K_ERR_UNSUPPORTED;
  const int b = bind_workspace(buf->bytes, scratch, kStaticScratchBytes);
  if (b != Q4K_OK) return b;
  // the arrival counters and tickets must start at zero; a launch that runs
  // to its end leaves them so, and this also covers one that never did
  if ((*cuda_err = cudaMemsetAsync(scratch, 0, h->counters, s)) != cudaSuccess) return Q4K_ERR_CUDA;
  return run_plan(buf->bytes, s, cuda_err);
}

}  // namespace q4k
