// q4k_gemv_seq: an ordered list of decode GEMV jobs y = W x (+ residual) over
// BLOCK144 Q4_K weights in one persistent launch (genie-ai-runtime §4,
// Path C: the GEMVs are the hot decode kernels and every decode step streams
// the whole model; §2: decode is bound by memory bandwidth).
//
// One CTA per SM stays resident for the whole list.  Its producer warp
// streams weights into a shared-memory ring and waits for nothing but free
// ring space, so the weight stream runs on across matrix boundaries and
// across the dependency points between jobs; 16 consumer warps dequantise
// and reduce.  This removes the launch gap, the start-up latency and the
// drain that separate launches pay at every matrix boundary.
//
// Segments.  Consecutive jobs that read the same x (same cols) form a
// segment.  A job with `wait` set starts a segment whose activations are read
// only after every earlier job has completed (a grid-wide arrival counter in
// the workspace); that is how a job consumes an earlier job's output inside
// the launch.  Only the activation reads wait: the weights of the waiting
// segment are already streaming into the ring.
//
// Work split.  A segment's rows (its jobs' rows, in order) are cut into
// equal contiguous runs, one per CTA (+-1 row), so every SM streams the same
// number of bytes whatever the matrix shape, and no row is shared between
// CTAs.  Rows of one job are contiguous in memory, so a stage of up to RS
// consecutive rows (about 24 KB, at least 8 rows) is ONE bulk copy: on GB300
// a bulk copy costs the copy engine a roughly fixed time, and copies of a
// few hundred bytes cannot reach the HBM rate while copies of 5 KB and more
// do.  Stages of varying size sit in a byte ring in shared memory, allocated
// and released in order.
//
// Consumers.  A unit is one group of 8 rows x 4 consecutive superblocks; a
// lane takes one row's whole superblock (256 weights), the 4 lanes of a row
// take the 4 superblocks, and the 8 rows of a warp read the same activations
// (shared-memory broadcast).  The 16 warps take a stage's units round-robin
// (continuing the rotation from stage to stage) and every warp visits every
// stage in order.  Each unit leaves one partial per row; after a pass of
// stages the CTA adds each row's partials in superblock order
// (deterministic), adds the residual and stores y.
//
// Arithmetic: 23-bit fixed-point activation planes and exact integer dp4a
// block sums, scales applied in fp32 (gemv_common.cuh).
#include "gemv_common.cuh"
#include "q4k_internal.h"
#include "tc_ptx.cuh"

#include <q4k.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

namespace q4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;   // + one producer warp
constexpr int kGroupRows = 8;               // rows of one warp unit (4 lanes per row)
constexpr int kStageTarget = 24576;         // bytes a stage aims at
constexpr int kMaxStageRows = 64;
constexpr int kNumBars = 16;                // stages in flight at most
constexpr size_t kSyncBytes = 256;

struct SeqJob {
  const uint8_t* w;
  const float* res;
  float* y;
  int rows;
  int row_base;     // first row of the job within its segment
};

struct SeqSeg {
  const float* x;
  int job_begin, job_end;
  int nb;           // superblocks per row
  int rows;         // rows of the segment
  int ctas;         // CTAs sharing its rows (<= grid, <= rows)
  int stage_rows;   // rows per full stage
  int pass_rows;    // rows per pass of partial sums
  int wait;         // read x only after every earlier segment has completed
};

struct SeqParams {
  SeqJob job[kGemvSeqMaxJobs];
  SeqSeg seg[kGemvSeqMaxJobs];
  int n_seg;
  int nb_max;
  int part_floats;
  int ring_bytes;
  unsigned* sync;     // [0] segment arrivals, [1] CTAs exited
  int* err;
};

struct SeqLayout {
  size_t xs, xss, part, ring, bars, total;
};

__host__ __device__ inline SeqLayout seq_layout(int B, int nb_max, int part_floats, int ring_bytes) {
  SeqLayout L;
  L.xs = 0;
  L.xss = L.xs + gemv::xs_bytes(B, nb_max);
  L.part = L.xss + gemv::xss_bytes(B, nb_max);
  L.ring = (L.part + sizeof(float) * (size_t)part_floats + 127) & ~size_t(127);
  L.bars = L.ring + (size_t)ring_bytes;
  L.total = L.bars + sizeof(uint64_t) * 2 * kNumBars + 16 + 1024;   // + flags, + base alignment slack
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

// The contiguous run of the segment's rows that CTA c owns.
__device__ __forceinline__ void cta_rows(const SeqSeg& S, int c, int& r0, int& r1) {
  if (c >= S.ctas) {
    r0 = r1 = 0;
    return;
  }
  r0 = (int)((long long)c * S.rows / S.ctas);
  r1 = (int)((long long)(c + 1) * S.rows / S.ctas);
}

__device__ __forceinline__ int job_of_row(const SeqParams& P, const SeqSeg& S, int r) {
  int j = S.job_begin;
  while (j + 1 < S.job_end && r >= P.job[j + 1].row_base) ++j;
  return j;
}

// The stage that starts at segment row r (< r1): its job and row count.
__device__ __forceinline__ int stage_at(const SeqParams& P, const SeqSeg& S, int r, int r1, int& jb) {
  jb = job_of_row(P, S, r);
  const SeqJob& J = P.job[jb];
  return min(S.stage_rows, min(r1, J.row_base + J.rows) - r);
}

// Byte position of the next stage in the ring: stages never wrap.
__device__ __forceinline__ uint32_t ring_place(uint32_t head, uint32_t bytes, uint32_t ring_bytes) {
  return head + bytes > ring_bytes ? 0u : head;
}

__device__ __forceinline__ void record_failure(const SeqParams& P) { atomicOr(P.err, 2); }

// Units of one stage for this warp: unit u is row group u / ng (8 rows) x
// superblock group u % ng (4 superblocks, ng = ceil(nb / 4)), and belongs to
// warp (base + u) % 16.  Lane (r, q) = (lane / 4, lane % 4) takes row r of
// the group and superblock 4*(u % ng) + q whole; the 4 lanes of a row add
// their superblocks ((s0 + s1) + (s2 + s3)) and lane q = 0 stores one
// partial per row and superblock group: part[row][group][b].
template <int B>
__device__ __forceinline__ void consume_stage(const uint8_t* stage, int n_rows, int nb, int base, float* part,
                                              int pass_row, const uint8_t* xs, const float2* xss, int warp,
                                              int lane) {
  const int ng = (nb + 3) >> 2;
  const int n_units = ((n_rows + kGroupRows - 1) / kGroupRows) * ng;
  const int r_in = lane >> 2, q = lane & 3;
  int u = (warp - base % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
  int g = u / ng, sg = u - g * ng;
  for (; u < n_units; u += kConsumerWarps) {
    const int row = g * kGroupRows + r_in, sb = sg * 4 + q;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    if (row < n_rows && sb < nb)
      gemv::superblock_dot<B, 4>(stage + ((size_t)row * nb + sb) * kBlockBytes, xs, xss, nb, sb, 0, acc);
#pragma unroll
    for (int b = 0; b < B; ++b) {
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
      acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
    }
    if (q == 0 && row < n_rows) {
#pragma unroll
      for (int b = 0; b < B; ++b) part[((size_t)(pass_row + row) * ng + sg) * B + b] = acc[b];
    }
    // next unit of this warp: 16 units on
    sg += kConsumerWarps;
    while (sg >= ng) {
      sg -= ng;
      ++g;
    }
  }
}

// Rows [pr0, pr0 + n) of the segment, partials part[row - pr0][group][b]:
// y = sum over superblock groups in order (+ residual).
template <int B>
__device__ __forceinline__ void reduce_pass(const SeqParams& P, const SeqSeg& S, int pr0, int n, const float* part,
                                            int tid) {
  const int ng = (S.nb + 3) >> 2;
  for (int i = tid; i < n * B; i += kConsumers) {
    const int rr = i / B, b = i - rr * B;
    const int r = pr0 + rr;
    const SeqJob& J = P.job[job_of_row(P, S, r)];
    const int row = r - J.row_base;
    const float* pp = part + (size_t)rr * ng * B + b;
    float v = 0.0f;
    for (int k = 0; k < ng; ++k) v += pp[(size_t)k * B];
    if (J.res) v += __ldcg(J.res + (size_t)b * J.rows + row);
    J.y[(size_t)b * J.rows + row] = v;
  }
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_seq_kernel(const __grid_constant__ SeqParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const SeqLayout L = seq_layout(B, P.nb_max, P.part_floats, P.ring_bytes);
  uint8_t* xs = smem + L.xs;
  float2* xss = reinterpret_cast<float2*>(smem + L.xss);
  float* part = reinterpret_cast<float*>(smem + L.part);
  uint8_t* ring = smem + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kNumBars;
  volatile int* flags = reinterpret_cast<volatile int*>(empty + kNumBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, grid = gridDim.x;
  const uint32_t ring_bytes = (uint32_t)P.ring_bytes;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], kConsumerWarps);
    }
    flags[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // in-flight stages [oldest, j); stage k occupies [pos_k, end_k) of the ring
      uint32_t spos[kNumBars], send[kNumBars];
      int j = 0, oldest = 0;
      uint32_t head = 0;
      bool ok = true;
      for (int si = 0; si < P.n_seg && ok; ++si) {
        const SeqSeg& S = P.seg[si];
        int r0, r1;
        cta_rows(S, c, r0, r1);
        const size_t row_bytes = (size_t)S.nb * kBlockBytes;
        for (int r = r0; r < r1 && ok;) {
          int jb;
          const int n = stage_at(P, S, r, r1, jb);
          const uint32_t bytes = (uint32_t)(n * row_bytes);
          const uint32_t pos = ring_place(head, bytes, ring_bytes);
          // release stages in order until none in flight overlaps the new
          // stage's bytes (after a wrap to 0 the oldest stage may lie in the
          // skipped tail while a younger one overlaps) and a barrier is free
          while (oldest < j) {
            bool busy = j - oldest >= kNumBars;
            for (int k = oldest; k < j && !busy; ++k)
              busy = pos < send[k % kNumBars] && spos[k % kNumBars] < pos + bytes;
            if (!busy) break;
            if (!tc::mbar_wait_sleep(&empty[oldest % kNumBars], (uint32_t)((oldest / kNumBars) & 1))) {
              ok = false;
              break;
            }
            ++oldest;
          }
          if (!ok) {
            record_failure(P);
            break;
          }
          const int slot = j % kNumBars;
          spos[slot] = pos;
          send[slot] = pos + bytes;
          const SeqJob& J = P.job[jb];
          tc::mbar_arrive_expect_tx(&full[slot], bytes);
          tc::bulk_g2s(ring + pos, J.w + (size_t)(r - J.row_base) * row_bytes, bytes, &full[slot]);
          head = pos + bytes;
          ++j;
          r += n;
        }
      }
      // every copy issued has landed before the CTA exits, even if consumers
      // gave up a wait and left early (bounded as well)
      for (int k = max(oldest, j - kNumBars); k < j; ++k)
        if (!tc::mbar_wait_sleep(&full[k % kNumBars], (uint32_t)((k / kNumBars) & 1))) record_failure(P);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  bool ok = true;
  const float* staged_x = nullptr;
  int staged_nb = -1;
  int j = 0;            // stage index in this CTA's ring order
  uint32_t head = 0;    // ring position, replayed exactly as the producer places stages
  int unit_base = 0;    // rotation of units over warps
  for (int si = 0; si < P.n_seg; ++si) {
    const SeqSeg& S = P.seg[si];
    int r0, r1;
    cta_rows(S, c, r0, r1);
    const int nb = S.nb;
    const size_t row_bytes = (size_t)nb * kBlockBytes;
    if (S.wait) {
      // activations may be outputs of earlier jobs: wait for all of them
      if (tid == 0 && ok && !grid_wait(P.sync, (unsigned)si * (unsigned)grid)) {
        record_failure(P);
        flags[0] = 1;
      }
      named_sync_consumers();
      ok = ok && !flags[0];
    }
    if (r1 > r0) {
      if (S.wait || S.x != staged_x || nb != staged_nb) {
        if (ok) gemv::stage_x<B, kConsumers, true>(S.x, nb, xs, xss, tid);
        staged_x = S.x;
        staged_nb = nb;
        named_sync_consumers();
      }
      int pass_r0 = r0, pass_n = 0;
      for (int r = r0; r < r1;) {
        int jb;
        const int n = stage_at(P, S, r, r1, jb);
        if (pass_n + n > S.pass_rows) {
          // partials of the pass are complete: reduce them
          if (!ok) flags[0] = 1;
          named_sync_consumers();
          ok = ok && !flags[0];
          if (ok) reduce_pass<B>(P, S, pass_r0, pass_n, part, tid);
          named_sync_consumers();
          pass_r0 = r;
          pass_n = 0;
        }
        const uint32_t bytes = (uint32_t)(n * row_bytes);
        const uint32_t pos = ring_place(head, bytes, ring_bytes);
        const int slot = j % kNumBars;
        if (ok && !tc::mbar_wait_sleep(&full[slot], (uint32_t)((j / kNumBars) & 1))) {
          ok = false;
          if (lane == 0) record_failure(P);
        }
        if (ok) consume_stage<B>(ring + pos, n, nb, unit_base, part, pass_n, xs, xss, warp, lane);
        // every warp releases every stage once, after its lanes read it
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[slot]);
        unit_base += ((n + kGroupRows - 1) / kGroupRows) * ((nb + 3) >> 2);
        head = pos + bytes;
        ++j;
        pass_n += n;
        r += n;
      }
      if (!ok) flags[0] = 1;
      named_sync_consumers();
      ok = ok && !flags[0];
      if (ok) reduce_pass<B>(P, S, pass_r0, pass_n, part, tid);
    }
    // every output of this CTA for the segment is stored: count the arrival
    named_sync_consumers();
    if (tid == 0) red_release_add_gpu(P.sync, 1u);
  }

  // the last CTA out resets the counters for the next launch
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.sync + 1, 1u) == (unsigned)grid - 1) {
      atomicExch(P.sync, 0u);
      atomicExch(P.sync + 1, 0u);
      __threadfence();
    }
  }
}

struct SeqPlan {
  int n_seg, nb_max, part_floats, ring_bytes, grid;
  size_t smem;
};

// Segments, CTA shares, stage and pass sizes of a job list.  Returns Q4K_OK or
// a status; fills P (if not null) and the plan.
int plan_seq(const q4k_gemv_job* jobs, int n_jobs, int B, const DeviceInfo& info, SeqParams* P,
             SeqPlan* plan) {
  if (n_jobs < 0 || n_jobs > kGemvSeqMaxJobs) return Q4K_ERR_UNSUPPORTED;
  SeqPlan p{};
  p.grid = info.sm_count;
  int n_seg = 0, n_job = 0;
  SeqSeg tseg[kGemvSeqMaxJobs];
  SeqJob tjob[kGemvSeqMaxJobs];
  bool pending_wait = false;
  const float* cur_x = nullptr;
  int cur_nb = -1;
  for (int i = 0; i < n_jobs; ++i) {
    const q4k_gemv_job& q = jobs[i];
    pending_wait = pending_wait || q.wait != 0;
    if (q.rows == 0) continue;
    const int nb = (int)(q.cols / kQK);
    if (n_seg == 0 || pending_wait || q.x != cur_x || nb != cur_nb) {
      if (n_seg > 0) tseg[n_seg - 1].job_end = n_job;
      SeqSeg s{};
      s.x = q.x;
      s.job_begin = n_job;
      s.nb = nb;
      s.wait = (pending_wait && n_seg > 0) ? 1 : 0;
      tseg[n_seg++] = s;
      cur_x = q.x;
      cur_nb = nb;
      pending_wait = false;
    }
    SeqJob jb{};
    jb.w = static_cast<const uint8_t*>(q.w);
    jb.res = q.residual;
    jb.y = q.y;
    jb.rows = (int)q.rows;
    tjob[n_job++] = jb;
  }
  if (n_seg > 0) tseg[n_seg - 1].job_end = n_job;
  p.n_seg = n_seg;
  p.nb_max = 1;
  size_t max_stage = 0;
  int min_part = 0;   // floats of the largest stage's partial sums
  for (int s = 0; s < n_seg; ++s) {
    SeqSeg& S = tseg[s];
    int64_t rows = 0;
    for (int j = S.job_begin; j < S.job_end; ++j) {
      tjob[j].row_base = (int)rows;
      rows += tjob[j].rows;
    }
    if (rows > (int64_t(1) << 30)) return Q4K_ERR_UNSUPPORTED;
    S.rows = (int)rows;
    S.ctas = (int)std::min<int64_t>(p.grid, rows);
    const int row_bytes = S.nb * kBlockBytes;
    const int rs = (kStageTarget / row_bytes) / kGroupRows * kGroupRows;
    S.stage_rows = std::max(kGroupRows, std::min(kMaxStageRows, rs));
    p.nb_max = std::max(p.nb_max, S.nb);
    max_stage = std::max(max_stage, (size_t)S.stage_rows * row_bytes);
    min_part = std::max(min_part, S.stage_rows * ((S.nb + 3) / 4) * B);
  }
  // shared memory: staged activations, then partial sums (up to a target,
  // at least one stage's worth), then a ring that holds two largest stages
  const size_t fixed = seq_layout(B, p.nb_max, 0, 0).total;
  if (fixed + 2 * max_stage + sizeof(float) * (size_t)min_part > (size_t)info.max_smem_optin)
    return Q4K_ERR_UNSUPPORTED;
  const size_t spare = (size_t)info.max_smem_optin - fixed - 2 * max_stage;
  const int target = B <= 2 ? 4096 : 8192;
  p.part_floats = (int)std::min<size_t>(target, spare / sizeof(float)) & ~31;
  if (p.part_floats < min_part) return Q4K_ERR_UNSUPPORTED;
  for (int s = 0; s < n_seg; ++s) tseg[s].pass_rows = p.part_floats / (((tseg[s].nb + 3) / 4) * B);
  const size_t with_part = seq_layout(B, p.nb_max, p.part_floats, 0).total;
  p.ring_bytes = (int)(((size_t)info.max_smem_optin - with_part) & ~size_t(127));
  p.smem = seq_layout(B, p.nb_max, p.part_floats, p.ring_bytes).total;
  if (p.smem > (size_t)info.max_smem_optin || (size_t)p.ring_bytes < 2 * max_stage) return Q4K_ERR_UNSUPPORTED;
  if (P) {
    std::memcpy(P->seg, tseg, sizeof(SeqSeg) * n_seg);
    std::memcpy(P->job, tjob, sizeof(SeqJob) * n_job);
    P->n_seg = n_seg;
    P->nb_max = p.nb_max;
    P->part_floats = p.part_floats;
    P->ring_bytes = p.ring_bytes;
  }
  *plan = p;
  return Q4K_OK;
}

template <int B>
cudaError_t launch_seq_b(const SeqParams& P, const SeqPlan& p, int dev, const DeviceInfo& info,
                         cudaStream_t s) {
  static int s_limit[64];
  int& limit = s_limit[dev & 63];
  if (limit < info.max_smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gemv_seq_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin);
    if (e != cudaSuccess) return e;
    limit = info.max_smem_optin;
  }
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

}  // namespace

int gemv_seq_workspace(const q4k_gemv_job* jobs, int n_jobs, int batch, size_t* bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
  SeqPlan p;
  const int st = plan_seq(jobs, n_jobs, batch, device_info(dev), nullptr, &p);
  if (st != Q4K_OK) return st;
  *bytes = kSyncBytes;
  return Q4K_OK;
}

int launch_gemv_seq(const q4k_gemv_job* jobs, int n_jobs, int batch, void* workspace, size_t workspace_bytes,
                    cudaStream_t s, cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  int dev = 0;
  if ((*cuda_err = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
  const DeviceInfo& info = device_info(dev);
  static thread_local SeqParams P;
  std::memset(&P, 0, sizeof(P));
  SeqPlan p;
  const int st = plan_seq(jobs, n_jobs, batch, info, &P, &p);
  if (st != Q4K_OK) return st;
  if (p.n_seg == 0) return Q4K_OK;
  if (workspace_bytes < kSyncBytes) return Q4K_ERR_INVALID_ARG;
  P.sync = static_cast<unsigned*>(workspace);
  P.err = device_error_word();
  if (!P.err) {
    *cuda_err = cudaGetLastError();
    return Q4K_ERR_CUDA;
  }
  cudaError_t e;
  switch (batch) {
    case 1: e = launch_seq_b<1>(P, p, dev, info, s); break;
    case 2: e = launch_seq_b<2>(P, p, dev, info, s); break;
    case 3: e = launch_seq_b<3>(P, p, dev, info, s); break;
    case 4: e = launch_seq_b<4>(P, p, dev, info, s); break;
    case 5: e = launch_seq_b<5>(P, p, dev, info, s); break;
    case 6: e = launch_seq_b<6>(P, p, dev, info, s); break;
    case 7: e = launch_seq_b<7>(P, p, dev, info, s); break;
    case 8: e = launch_seq_b<8>(P, p, dev, info, s); break;
    default: return Q4K_ERR_UNSUPPORTED;
  }
  *cuda_err = e;
  return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

}  // namespace q4k
