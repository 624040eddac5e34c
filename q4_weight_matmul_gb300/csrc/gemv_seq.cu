// q4k_gemv_seq: the host side of the persistent job-list GEMV (planning,
// prepared plans, the allocation-free entry); the kernel is in
// gemv_seq_kernel.cuh.
#include "gemv_seq_kernel.cuh"

#include <mutex>

namespace q4k {
namespace seq {
Q4K_SEQ_VARIANTS(Q4K_SEQ_DECLARE, false)
Q4K_SEQ_VARIANTS(Q4K_SEQ_DECLARE, true)
}  // namespace seq

namespace {
using namespace seq;

struct SeqPlan {
  int n_seg, n_epoch, nb_max, ring, part_floats, grid;
  int q6;   // holds Q6_K jobs
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
// Units per CTA from which an epoch counts as long (see the pass size below).
constexpr int64_t kLongEpochUnitsPerCta = 64;

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
  // shared memory: activations, partial sums, then the deepest ring that fits.
  // At batch 1 a launch whose epochs are long (many units per CTA) takes
  // passes of 256 units, which keeps the reduction syncs rare; one whose
  // epochs are short (engine-order layers, a single decode set) takes passes
  // of 32 units and gives the memory to 3 more ring slots, which shortens
  // the latency-bound epochs (measured: 13-set launch -6.5 % with short
  // passes; decode layer with waits -3.3 %, token -3.4 % with them).
  int64_t max_per_cta = 0;
  for (int e = 0; e < n_epoch; ++e) max_per_cta = std::max<int64_t>(max_per_cta, (tep[e].units + p.grid - 1) / p.grid);
  const int b1_mult = max_per_cta >= kLongEpochUnitsPerCta ? 16 : 2;
  p.part_floats = 16 * kRB * B * (B == 1 ? b1_mult : (B == 2 ? 8 : (B <= 4 ? 2 : 1)));
  p.ring = 0;
  const int slot_bytes = n_q6 > 0 ? kQ6UnitBytes : kUnitBytes;
  p.q6 = n_q6 > 0;
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
    cudaError_t e = set_smem<B, false>(info.max_smem_optin);
    if (e != cudaSuccess) return e;
    e = set_smem<B, true>(info.max_smem_optin);
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
  return p.q6 ? launch<B, true>(P, (unsigned)p.grid, p.smem, s) : launch<B, false>(P, (unsigned)p.grid, p.smem, s);
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

// Q4K_OK when `buf` holds a plan written by gemv_seq_plan on the current device.
int check_plan(const void* buf, cudaError_t* ce) {
  *ce = cudaSuccess;
  const PlanHeader* h = static_cast<const PlanHeader*>(buf);
  if (h->magic != kPlanMagic || !h->ws) return Q4K_ERR_INVALID_ARG;
  int dev = 0;
  if ((*ce = cudaGetDevice(&dev)) != cudaSuccess) return Q4K_ERR_CUDA;
  if (dev != h->dev) return Q4K_ERR_INVALID_ARG;
  return Q4K_OK;
}

int run_plan(const void* buf, cudaStream_t s, cudaError_t* ce) {
  if (const int st = check_plan(buf, ce)) return st;
  const PlanHeader* h = static_cast<const PlanHeader*>(buf);
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

int gemv_seq_check_plan(const void* plan, cudaError_t* cuda_err) { return check_plan(plan, cuda_err); }

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
