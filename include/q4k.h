/*
 * q4k.h - C ABI of libq4k.so, the GB300 (sm_103a) Q4_K weight-matmul library.
 *
 * The library computes the Q4_K-quantised weight matmul of an LLM inference
 * engine in its two halves (genie-ai-runtime: a Jetson edge LLM inference
 * engine, §2 "the roofline that dictates strategy"): the bandwidth-bound
 * decode GEMV and the compute-bound prefill GEMM over q8_1 activations.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All data pointers are DEVICE pointers (cudaMalloc'd or torch-owned) on
 *    the current CUDA device.  The caller owns every buffer; the library never
 *    allocates, frees or retains a caller pointer after the call returns.
 *  - `stream` is a cudaStream_t passed as `void*` (NULL = legacy default
 *    stream).  Every compute call only validates its arguments on the host
 *    and enqueues work on `stream`; it returns before the GPU finishes.
 *  - A non-zero return value is a `q4k_status`; when a call returns anything
 *    but Q4K_OK nothing was enqueued (Q4K_ERR_CUDA: a launch failed and the
 *    CUDA error string is available from q4k_last_error_string()).
 *  - Matrices are row-major.  A weight matrix W has `rows` outputs and `cols`
 *    inputs; `cols` must be a positive multiple of 256 (one superblock).
 *    Activations are [tokens][cols], outputs are [tokens][rows].
 *  - Device pointers must be 16-byte aligned (Q4K_ERR_ALIGNMENT otherwise).
 *  - Sizes of zero (rows, tokens, batch) are valid and enqueue nothing.
 *  - A call whose work takes more than one kernel launch (a q4k_gemv_seq
 *    list of more than 96 jobs, or 48 Q6_K jobs) validates and plans all of
 *    it first; only a
 *    CUDA launch failure of a later launch can leave the earlier ones
 *    enqueued (the status is then Q4K_ERR_CUDA).
 *
 * Accuracy of every fp32 output (decode GEMV and prefill GEMM).  The kernels
 * apply the scale term d*sc*q and the min term dmin*m of each weight as
 * separate sums, as the MMQ form does, so their rounding is bounded against
 *     M = sum_k (|d*sc*q_k| + |dmin*m_k|) * |x_k|   (+ |residual|):
 *     |y - exact| <= 1e-4 * M,
 * where x is the fp32 activation (GEMV) or the dequantised q8_1 activation
 * d8*q8 (GEMM).  M equals sum_k |w_k||x_k| except where the two terms of a
 * weight cancel, and the bound is then also 1e-4 * sum_k |w_k||x_k|
 * whenever M <= 1.5 * sum_k |w_k||x_k|.  The bound holds for finite inputs
 * whose nonzero products |d*sc*q*x|, |dmin*m*x| and results lie between
 * 2^-100 and 2^100 (nearer fp32's underflow or overflow, its own rounding
 * there bounds the error instead).
 *
 * The Q4_K superblock (genie-ai-runtime §2 "Qwen3-4B Q4_K_M weights"; the
 * pages name the format but print no byte layout, so the common GGUF Q4_K
 * byte order is used): 256 weights with an fp16 scale d and an fp16 min
 * dmin, eight 32-weight sub-blocks with a 6-bit scale sc and a 6-bit min m,
 * and a 4-bit quant q per weight; each weight is w = d*sc*q - dmin*m.
 * Q4K_LAYOUT_BLOCK144 stores each superblock in 144 bytes: d (2 bytes,
 * little-endian binary16), dmin (2), 12 packed scale/min bytes, 128 quant
 * bytes (weight 64c+l in the low nibble and 64c+32+l in the high nibble of
 * byte 32c+l).  W occupies rows * (cols/256) * 144 bytes, superblocks of a
 * row contiguous, rows contiguous.
 */
#ifndef Q4K_H
#define Q4K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum q4k_status {
  Q4K_OK = 0,
  Q4K_ERR_INVALID_ARG = 1,    /* null pointer, bad size or shape           */
  Q4K_ERR_ALIGNMENT = 2,      /* a pointer is not 16-byte aligned          */
  Q4K_ERR_UNSUPPORTED = 3,    /* a valid request this build does not serve */
  Q4K_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed      */
  Q4K_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up a bounded wait           */
} q4k_status;

typedef enum q4k_layout {
  Q4K_LAYOUT_BLOCK144 = 0,    /* 144-byte superblocks, GGUF byte order     */
  Q4K_LAYOUT_GPU = 1          /* reserved: rows interleaved for vector
                                 loads; every call returns
                                 Q4K_ERR_UNSUPPORTED (see below)           */
} q4k_layout;

/*
 * Q4K_LAYOUT_GPU is the row-interleaved repack that CPU kernels use to load
 * several rows per vector ("I'm making LLMs work on small and old devices":
 * the llama.cpp repack of row counts divisible by 8).  This library does not
 * build it: its kernels copy BLOCK144 weights with 3-D tensor copies whose
 * boxes already regroup rows (row r of a 32-row box is 144 bytes from row
 * r+1 in shared memory), so an interleaved copy in device memory would gain
 * nothing and cost a second layout.
 */

/* Bytes of a packed rows x cols weight matrix in `layout`
 * (rows * cols/256 * 144 for BLOCK144); 0 for an invalid or unsupported
 * request.  (genie-ai-runtime §2: Qwen3-4B Q4_K_M weights, ~2.3 GB, are
 * what every decode step streams.) */
size_t q4k_packed_bytes(int64_t rows, int64_t cols, int layout);

/*
 * q4k_pack - pack Q4_K fields into superblocks (the packer/layout step;
 * genie-ai-runtime §2 names the Q4_K_M format the engine runs; the byte
 * order is the one described at the top of this header).
 *   d, dmin : uint16 binary16 bits, [rows][cols/256]
 *   sc, m   : uint8 values 0..63,   [rows][cols/32]   (bits above 5 ignored)
 *   q       : uint8 values 0..15,   [rows][cols]      (bits above 3 ignored)
 *   w       : output, q4k_packed_bytes(rows, cols, layout) bytes
 * Bit-exact: the result depends only on the input bits.
 */
int q4k_pack(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc,
             const uint8_t* m, const uint8_t* q, int64_t rows, int64_t cols,
             int layout, void* w, void* stream);

/*
 * q4k_unpack - test export, the inverse of q4k_pack: read every field back
 * out of packed superblocks (same arrays and shapes as q4k_pack; sc, m and q
 * come back in their low 6 / 6 / 4 bits with the bits above them zero).
 * Bit-exact: q4k_unpack(q4k_pack(f)) == f for fields within their ranges.
 */
int q4k_unpack(const void* w, int layout, int64_t rows, int64_t cols,
               uint16_t* d, uint16_t* dmin, uint8_t* sc, uint8_t* m,
               uint8_t* q, void* stream);

/*
 * q8_1_bytes - device bytes of the q8_1 form of a tokens x cols activation
 * matrix: q (1 byte per element) plus d8 and sum (4 bytes each per 32
 * elements), whether kept in one buffer or three; 0 for an invalid request.
 */
size_t q8_1_bytes(int64_t tokens, int64_t cols);

/*
 * q8_quantize - fp32 activations to q8_1 blocks of 32 (prefill input: the
 * integer activation blocks of the MMQ form; genie-ai-runtime §3 Path E is
 * the batched Q4_K prefill kernel these feed; the pages do not print the
 * block, so its definition is this one).
 * For each row t and each block b of 32 consecutive columns:
 *   amax = max |x|, d8 = amax / 127 (IEEE fp32 division),
 *   q = clamp(roundf(x / d8), -127, 127) (fp32 division, ties away from 0),
 *   sum = sum of the 32 q; a block whose d8 is 0 gives q = 0, sum = 0.
 *   x   : float [tokens][cols]   (cols a multiple of 256)
 *   q   : int8  [tokens][cols]
 *   d8  : float [tokens][cols/32]
 *   sum : int32 [tokens][cols/32]
 * Bit-exact.  Non-finite inputs give unspecified (but in-bounds) output.
 */
int q8_quantize(const float* x, int64_t tokens, int64_t cols, int8_t* q,
                float* d8, int32_t* sum, void* stream);

/*
 * q8_quantize_h16 - q8_quantize with the quants stored as binary16 values
 * (every q is an integer in [-127, 127], exact in binary16): the operand
 * form the tensor cores read, so q4k_gemm_h16 loads it without converting.
 *   q : uint16 binary16 bits [tokens][cols]; d8, sum as for q8_quantize.
 * Bit-exact: q holds exactly the values q8_quantize writes, d8 and sum are
 * the same bits.
 */
int q8_quantize_h16(const float* x, int64_t tokens, int64_t cols, uint16_t* q,
                    float* d8, int32_t* sum, void* stream);

/*
 * q4k_gemv - decode GEMV (genie-ai-runtime §4, Path C: the hot decode
 * kernels; residual add folded into the GEMV):
 *   y[b][o] = sum_k w[o][k] * x[b][k]  (+ residual[b][o] if residual != NULL)
 *   w        : packed weights (layout), rows x cols
 *   x        : float [batch][cols], 1 <= batch <= 8
 *   residual : float [batch][rows] or NULL
 *   y        : float [batch][rows]; may alias residual, not x or w
 * Accuracy: the bound at the top of this header, per element.
 * Arithmetic: each 32-wide block of x is held as a 32-bit fixed-point
 * integer with a power-of-two scale, the quant-times-x block sums are exact
 * integers, and the scales d*sc, dmin*m are applied in fp32.  Blocks where
 * 24 bits keep every element within 2^-14 of itself use three byte planes,
 * blocks that need more add a fourth, and blocks that 32 bits cannot hold
 * that closely (an element below ~2^-16 of the block's largest, or a
 * largest |x| outside [2^-87, 2^94)) are summed in fp32.
 * Deterministic: the same inputs give the same bits on every run.
 */
int q4k_gemv(const void* w, int layout, int64_t rows, int64_t cols,
             const float* x, int64_t batch, const float* residual, float* y,
             void* stream);

/*
 * q4k_gemv_q8 - the MMQ product for a few tokens as a GEMV: batch (1..8)
 * rows of q8_1 activations against one weight matrix, in one weight pass
 * (genie-ai-runtime §3: prompts of 18-33 tokens are the engine's prefill
 * regime, far below a tensor-core tile; batched decode and speculative
 * verification of a few tokens are the same shape).
 *   y[b][o] = sum_blk ( d*sc * d8[b,blk] * P[b,o,blk] - dmin*m * d8[b,blk]*sum[b,blk] )
 *             (+ residual[b][o] if residual != NULL),
 *   P = exact integer dot of the 32 quants with the 32 int8 q8 values.
 *   q8, d8, sum : q8_quantize() output for `batch` rows of width cols
 *   y           : float [batch][rows]; residual as for q4k_gemv
 * Accuracy as q4k_gemm (the bound at the top of this header, x = d8*q8).
 * q4k_gemm and q4k_gemm_h16 use this kernel for up to 32 tokens (a launch
 * per 8 tokens), and their block-dot exports then come from it.
 */
int q4k_gemv_q8(const void* w, int layout, int64_t rows, int64_t cols,
                const int8_t* q8, const float* d8, const int32_t* sum,
                int64_t batch, const float* residual, float* y, void* stream);

/*
 * q4k_gemv_multi - one decode GEMV launch over n (1..4) matrices that share
 * the input x (genie-ai-runtime §4, Path C: one kernel for the QKV triple and
 * for the gate/up pair).  w, rows, y (and residual, if not NULL) are HOST
 * arrays of n entries; entry m is a q4k_gemv problem with its own device
 * pointers w[m], y[m], residual[m] (nullable) and row count rows[m].  All
 * matrices have `cols` inputs.  Matrices with rows[m] == 0 are skipped.
 * Same accuracy and determinism as q4k_gemv; n > 4 gives Q4K_ERR_UNSUPPORTED.
 */
int q4k_gemv_multi(int n, const void* const* w, int layout, const int64_t* rows,
                   int64_t cols, const float* x, int64_t batch,
                   const float* const* residual, float* const* y, void* stream);

/*
 * q4k_gemv_job - one decode GEMV of a q4k_gemv_seq list:
 *   y[b][o] = sum_k w[o][k] * x[b][k]  (+ residual[b][o] if residual != NULL)
 */
typedef struct q4k_gemv_job {
  const void* w;           /* packed weights (layout), rows x cols              */
  int64_t rows;            /* outputs; a job with 0 rows is skipped             */
  int64_t cols;            /* inputs, a positive multiple of 256                */
  const float* x;          /* float [batch][cols]                               */
  const float* residual;   /* float [batch][rows] or NULL                       */
  float* y;                /* float [batch][rows]; may alias residual           */
  int32_t wait;            /* non-zero: x and residual are read only after every
                              earlier job of the list has stored its y          */
  int32_t format;          /* 0: Q4_K weights in the call's `layout`;
                              1: Q6_K weights in Q6K_LAYOUT_GPU (the Q6_K
                              superblock dot of q6k_gemv and its accuracy)     */
} q4k_gemv_job;

#define Q4K_GEMV_SEQ_MAX_JOBS 256

/*
 * q4k_gemv_seq_workspace_bytes - device workspace that q4k_gemv_seq needs for
 * this job list and batch on the current device (it depends on where the
 * list's `wait` flags fall, on the batch and on the SM count); 0 when the
 * request is invalid or unsupported.
 */
size_t q4k_gemv_seq_workspace_bytes(const q4k_gemv_job* jobs, int n_jobs, int64_t batch);

/*
 * q4k_gemv_seq - an ordered list of decode GEMVs in ONE persistent launch
 * per 96 jobs, 48 of them Q6_K at most (genie-ai-runtime §4, Path C: the GEMVs are the hot decode
 * kernels, and every decode step streams the whole model's weights; §2:
 * decode is bound by memory bandwidth).  One CTA per SM streams the weights
 * of job after job without a launch boundary, each SM the same share of the
 * bytes between two `wait` points; a job with `wait` set reads its activations
 * only after every earlier job has completed, so it may consume an earlier
 * job's y (a decode layer: QKV | o | gate,up | down, each waiting on the
 * previous).  Jobs between two `wait` points may run concurrently: none of
 * them may read what another of them writes.
 *   jobs      : HOST array of n_jobs (0..Q4K_GEMV_SEQ_MAX_JOBS) entries, read
 *               during the call only; device pointers as in q4k_gemv
 *   batch     : 1..8 activation rows per job (0: nothing to do)
 *   workspace : device memory of at least q4k_gemv_seq_workspace_bytes()
 *               bytes, 16-byte aligned, zero-filled before its first use
 *               (e.g. cudaMemset).  It holds the launch's arrival
 *               counters and tickets, which each call resets before it ends
 *               (also when its kernel gave up a bounded wait), and the
 *               partial row sums of row blocks that CTAs share, which need
 *               no clearing; the workspace is reused as it is.  Calls that
 *               share a workspace must not overlap on the GPU.
 * The launch is cooperative (every CTA resident at once, one per SM); it
 * fails with Q4K_ERR_CUDA when the GPU cannot hold them all.
 * Jobs may mix Q4_K and Q6_K weights (q4k_gemv_job.format): a Q4_K_M
 * layer, whose down and v projections are Q6_K in half the layers, runs as
 * one list.  Accuracy and arithmetic as q4k_gemv (Q6_K jobs: as q6k_gemv).
 * Deterministic: for one job list on one device, the same inputs give the
 * same bits on every run.
 * Errors: Q4K_ERR_INVALID_ARG (null pointer, bad size, workspace too small),
 * Q4K_ERR_ALIGNMENT, Q4K_ERR_UNSUPPORTED (more jobs than the maximum, batch
 * above 8, activations too wide to stage in shared memory).
 */
int q4k_gemv_seq(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * q4k_gemv_seq_plan / q4k_gemv_seq_launch - q4k_gemv_seq split into a
 * planning step done once and a launch done every step, for an engine that
 * runs the same job list with the same buffers every decode step (the pages'
 * engine pre-allocates its pools and does no allocation or set-up on the
 * hot path, genie-ai-runtime §4 "Memory-first").
 *   plan_bytes = q4k_gemv_seq_plan_bytes(n_jobs): host bytes of a plan
 *     (room for one launch of about 28 KB per 48 jobs, the most Q6_K jobs
 *     one launch takes); 0 if n_jobs is out of range.
 *   q4k_gemv_seq_plan validates the list exactly as q4k_gemv_seq does and
 *     writes the plan (tensor maps of every weight matrix, the work split,
 *     every device pointer of the jobs and the workspace) into `plan`:
 *     caller-owned HOST memory of at least plan_bytes bytes, 64-byte
 *     aligned (Q4K_ERR_ALIGNMENT otherwise).  It enqueues nothing and
 *     allocates nothing; `workspace` is as for q4k_gemv_seq.
 *   q4k_gemv_seq_launch enqueues the plan's launches on `stream`: the same
 *     work, results and accuracy as the q4k_gemv_seq call the plan was made
 *     from.  The pointers baked into the plan must stay valid, the plan must
 *     not be changed, and launches from one plan (or of plans sharing a
 *     workspace) must not overlap on the GPU.  Call it on the device that was
 *     current when the plan was made (Q4K_ERR_INVALID_ARG otherwise).
 */
size_t q4k_gemv_seq_plan_bytes(int n_jobs);
int q4k_gemv_seq_plan(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch,
                      void* workspace, size_t workspace_bytes, void* plan, size_t plan_bytes);
int q4k_gemv_seq_launch(const void* plan, void* stream);

/*
 * q4k_gemv_seq_launch_host - one decode step from HOST buffers, for an
 * engine whose activations live on the host between steps (the pages'
 * engine keeps its buffers allocated for the whole run and only moves data
 * on the hot path, genie-ai-runtime §4 "Memory-first"): enqueues on
 * `stream`, in order, the copy of x_bytes bytes from x_host to x_dev, the
 * plan's launches (as q4k_gemv_seq_launch) and the copy of y_bytes bytes
 * from y_dev to y_host, and returns without waiting; y_host holds the
 * step's outputs once the stream has reached that point (synchronise the
 * stream before reading it).  x_dev and y_dev are device buffers that the
 * caller laid out to hold the jobs' inputs and outputs (the plan's x and y
 * pointers are views into them); the library cannot check that.  Host
 * buffers should be pinned (page-locked), or the copies are not
 * asynchronous.  A zero byte count skips that copy.
 * Errors: Q4K_ERR_INVALID_ARG (null plan, or a null pointer with a non-zero
 * byte count, or a plan made on another device) with nothing enqueued;
 * Q4K_ERR_CUDA if an enqueue fails, after which the steps before it stay
 * enqueued.
 */
int q4k_gemv_seq_launch_host(const void* plan, const void* x_host, void* x_dev, size_t x_bytes,
                             void* y_host, const void* y_dev, size_t y_bytes, void* stream);

/*
 * q4k_gemv_seq_static - q4k_gemv_seq for callers that cannot allocate device
 * memory: a serving process that fixes its device memory at start-up and may
 * not allocate afterwards, a plug-in that runs inside a host program whose
 * allocator it may not touch, or plain C code with no allocator at all.  The
 * pages have no counterpart; it is an addition for such callers.
 * Same jobs, batch, layout, results and accuracy as q4k_gemv_seq, but no
 * workspace argument: the scratch is a fixed 1 MiB array in the library's
 * device memory, which every GPU that loads the library holds until the
 * process exits.  The call itself allocates nothing (no cudaMalloc, no
 * allocating library routine).
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and keeps it; make that first call before any
 *    stream capture.
 *  - Each call plans and checks the whole list first, then clears the
 *    array's counters on `stream`, then launches; if that launch fails,
 *    the clear (of the library's own array) is the one thing left enqueued.
 *  - All calls on a device share the one array: calls that overlap on the
 *    GPU (other streams, other host threads) race and give wrong results.
 *  - A job list whose scratch would exceed 1 MiB (the need grows with the
 *    batch and the SM count; a GB300 at batch 8 needs about 0.6 MiB) gives
 *    Q4K_ERR_UNSUPPORTED and enqueues nothing.
 */
int q4k_gemv_seq_static(const q4k_gemv_job* jobs, int n_jobs, int layout, int64_t batch,
                        void* stream);

/*
 * q4k_gemm - prefill MMQ GEMM (genie-ai-runtime §3, "The tensor-core kernel
 * (Path E)"; integer form over q8_1 activations):
 *   y[t][o] = sum_b ( d*sc[o,b] * d8[t,b] * P[t,o,b]
 *                     - dmin*m[o,b] * d8[t,b] * sum[t,b] ),
 *   P[t,o,b] = sum_{i<32} q[o][32b+i] * q8[t][32b+i]   (exact integers)
 *   w         : packed weights (layout), rows x cols
 *   q8,d8,sum : q8_quantize() output for `tokens` rows of width cols
 *   y         : float [tokens][rows]
 * Accuracy: the bound at the top of this header, with x = d8*q8.
 */
int q4k_gemm(const void* w, int layout, int64_t rows, int64_t cols,
             const int8_t* q8, const float* d8, const int32_t* sum,
             int64_t tokens, float* y, void* stream);

/*
 * q4k_gemm_h16 - q4k_gemm over q8_quantize_h16 output (the same MMQ form,
 * results and accuracy); the fast prefill path: tensor copies load the
 * binary16 quants straight into the tensor cores' operand layout.
 *   q16 : uint16 binary16 quants [tokens][cols] (values -127..127)
 * Other arguments as for q4k_gemm.
 */
int q4k_gemm_h16(const void* w, int layout, int64_t rows, int64_t cols,
                 const uint16_t* q16, const float* d8, const int32_t* sum,
                 int64_t tokens, float* y, void* stream);

/*
 * x_split_f16 / q4k_gemm_f16 - the prefill GEMM in the fp16-operand form of
 * genie-ai-runtime §3, "The tensor-core kernel (Path E)" (fp16 activations,
 * fp32 accumulation), computing the product with the dequantised weights
 * and fp32 activations directly (no q8_1 step):
 *   y[t][o] = sum_k w[o][k] * x[t][k]
 * x_split_f16 prepares the activations once per input (shared by every
 * matrix that reads it): each token row t gets a power-of-two scale s_t
 * that puts its largest |x| in [2^14, 2^15), and each X = s_t * x is held
 * as hi = fp16(X) and lo = fp16(X - hi).
 *   x         : float [tokens][cols]
 *   hi, lo    : uint16 binary16 [tokens][cols]
 *   bsum      : uint16 binary16 [tokens][cols/256][16]: per superblock the
 *               eight 32-wide block sums of hi + lo, times 2^-6, as hi parts
 *               then lo parts
 *   inv_scale : float [tokens], 1/s_t
 * x_split_f16_bytes gives the bytes of all four arrays together (0 for an
 * invalid request).  q4k_gemm_f16 then runs the tensor-core GEMM over the
 * split activations (any tokens >= 1; rows and cols as q4k_gemm):
 *   y : float [tokens][rows]
 * Accuracy: |y - exact| <= 1e-4 * (M + 2^-16 * max_k|x_k| * W1) per element,
 * M the norm at the top of this header (fp32 x) and
 * W1 = sum_k (|d*sc*q_k| + |dmin*m_k|): the hi/lo pair keeps each element
 * to 2^-22 of itself, and elements below about 2^-24 of their row's largest
 * are rounded in absolute terms (the second term).  Range as at the top of
 * this header, for rows whose largest |x| lies in [2^-110, 2^110].
 */
size_t x_split_f16_bytes(int64_t tokens, int64_t cols);
int x_split_f16(const float* x, int64_t tokens, int64_t cols, uint16_t* hi,
                uint16_t* lo, uint16_t* bsum, float* inv_scale, void* stream);
int q4k_gemm_f16(const void* w, int layout, int64_t rows, int64_t cols,
                 const uint16_t* hi, const uint16_t* lo, const uint16_t* bsum,
                 const float* inv_scale, int64_t tokens, float* y, void* stream);

/*
 * q4k_gemm_blockdots - test export of the GEMM's per-block integer dots,
 * computed by the same tensor-core main loop as q4k_gemm:
 *   p[t][o][b] = sum_{i<32} q[o][32b+i] * q8[t][32b+i]
 *   p : int32 [tokens][rows][cols/32]
 * Bit-exact.
 */
int q4k_gemm_blockdots(const void* w, int layout, int64_t rows, int64_t cols,
                       const int8_t* q8, int64_t tokens, int32_t* p,
                       void* stream);

/* q4k_gemm_blockdots_h16 - the same test export from q4k_gemm_h16's main
 * loop (binary16 quants q16 as for q4k_gemm_h16).  Bit-exact. */
int q4k_gemm_blockdots_h16(const void* w, int layout, int64_t rows, int64_t cols,
                           const uint16_t* q16, int64_t tokens, int32_t* p,
                           void* stream);

/*
 * Q6_K weights (genie-ai-runtime §2: Q4_K_M models keep some matrices in
 * Q6_K; §6 "The negatives I kept", Path G: a Q6_K block layout redesigned
 * for vectorised loads is the open attack on Q6_K decode).  The pages print
 * no Q6_K layout; the common GGUF Q6_K block is used: 256 weights with a
 * binary16 scale d, sixteen int8 scales sc (one per 16 weights) and a 6-bit
 * quant q per weight, w = d * sc * (q - 32).
 *  - Q6K_LAYOUT_GGUF: 210-byte superblocks in GGUF byte order (ql[128] low
 *    nibbles, qh[64] high bit pairs, scales[16], d), rows * cols/256 * 210
 *    bytes.  210 is not a multiple of 16, so superblocks do not start on
 *    16-byte boundaries and no tensor copy can fetch them: the GEMV does not
 *    read this layout (Q4K_ERR_UNSUPPORTED); convert it with q6k_repack.
 *  - Q6K_LAYOUT_GPU: per row, the row's superblocks as 208-byte blocks (the
 *    16 scales, then per 64 weights 32 bytes of low nibbles and 16 bytes of
 *    high bit pairs), then the row's d values, then zero padding to a
 *    multiple of 16 bytes: rows * roundup16(cols/256 * 210) bytes, so the
 *    padding is under 16 bytes a row.  The exact byte order is defined by
 *    q6k_pack and read back by q6k_unpack.
 */
typedef enum q6k_layout {
  Q6K_LAYOUT_GGUF = 0,
  Q6K_LAYOUT_GPU = 1
} q6k_layout;

/* Bytes of a rows x cols Q6_K matrix in `layout`; 0 for an invalid request. */
size_t q6k_packed_bytes(int64_t rows, int64_t cols, int layout);

/*
 * q6k_pack - pack Q6_K fields into `layout`:
 *   d  : uint16 binary16 bits, [rows][cols/256]
 *   sc : int8,                 [rows][cols/16]
 *   q  : uint8 values 0..63,   [rows][cols]   (bits above 5 ignored)
 *   w  : output, q6k_packed_bytes(rows, cols, layout) bytes
 * Bit-exact.  Every pointer 16-byte aligned.
 */
int q6k_pack(const uint16_t* d, const int8_t* sc, const uint8_t* q, int64_t rows,
             int64_t cols, int layout, void* w, void* stream);

/*
 * q6k_repack - convert packed Q6_K weights between layouts (a loader that
 * reads GGUF blocks from a file calls it once per matrix with
 * src_layout = Q6K_LAYOUT_GGUF, dst_layout = Q6K_LAYOUT_GPU).  src and dst
 * must not overlap.  Bit-exact; a GGUF source needs only 2-byte alignment
 * (its blocks are 210 bytes), every other pointer 16-byte alignment.
 */
int q6k_repack(const void* src, int src_layout, int64_t rows, int64_t cols,
               void* dst, int dst_layout, void* stream);

/*
 * q6k_unpack - test export, the inverse of q6k_pack (fields as for
 * q6k_pack; q comes back in its low 6 bits).  Alignment as for q6k_repack.
 */
int q6k_unpack(const void* w, int layout, int64_t rows, int64_t cols,
               uint16_t* d, int8_t* sc, uint8_t* q, void* stream);

/*
 * q6k_gemv - decode GEMV over Q6_K weights in Q6K_LAYOUT_GPU (the same
 * kernel as q4k_gemv, with the Q6_K superblock dot):
 *   y[b][o] = sum_k w[o][k] * x[b][k]  (+ residual[b][o] if residual != NULL)
 *   w        : Q6K_LAYOUT_GPU weights, rows x cols
 *   x        : float [batch][cols], 1 <= batch <= 8
 *   residual : float [batch][rows] or NULL
 *   y        : float [batch][rows]; may alias residual, not x or w
 * Accuracy: |y - exact| <= 1e-4 * (sum_k |w_k||x_k| + |residual|) per
 * element, under the range condition at the top of this header (the quant
 * enters the integer dot as the signed q - 32, so there is no second term).
 * Arithmetic and determinism as q4k_gemv.  Q4K_ERR_UNSUPPORTED for a GGUF
 * layout, batch > 8, or a shape whose staged activations do not fit.
 */
int q6k_gemv(const void* w, int layout, int64_t rows, int64_t cols,
             const float* x, int64_t batch, const float* residual, float* y,
             void* stream);

/*
 * q6k_gemv_q8 / q6k_gemm - the MMQ product over Q6_K weights (Q6K_LAYOUT_GPU)
 * and q8_1 activations (q8_quantize output; the block sums may be NULL, the
 * Q6_K product has no min term):
 *   y[t][o] = sum_g (d*sc_g)[o] * d8[t][g/2] * P[t][o][g]   (+ residual[t][o])
 *   P[t][o][g] = sum_{i<16} (q[o][16g+i] - 32) * q8[t][16g+i]   (exact integers)
 * q6k_gemv_q8 takes 1..8 token rows in one weight pass (batch decode, short
 * prompts); q6k_gemm takes any token count as launches of up to 8 token rows
 * each (the weights are read once per 8 tokens: the prefill of a few tokens
 * and short prompts, not a tensor-core GEMM).  y: float [tokens][rows].
 * Accuracy: |y - exact| <= 1e-4 * sum_k |w_k| |d8*q8_k| (+ |residual|).
 * Deterministic.  All launches' shapes are checked before the first is
 * enqueued.
 */
int q6k_gemv_q8(const void* w, int layout, int64_t rows, int64_t cols,
                const int8_t* q8, const float* d8, const int32_t* sum,
                int64_t batch, const float* residual, float* y, void* stream);
int q6k_gemm(const void* w, int layout, int64_t rows, int64_t cols,
             const int8_t* q8, const float* d8, const int32_t* sum,
             int64_t tokens, float* y, void* stream);

/*
 * q6k_gemm_f16 - the fp16-activation tensor-core prefill GEMM (as
 * q4k_gemm_f16) over Q6K_LAYOUT_GPU weights, on x_split_f16 output (bsum may
 * be NULL: the Q6_K product has no min term):
 *   y[t][o] = sum_k w[o][k] * x[t][k],   w = d * sc * (q - 32)
 * Accuracy: |y - exact| <= 1e-4 * (sum_k |w_k||x_k| + 2^-16 * max_k|x_k| *
 * sum_k |w_k|) per element (the split's bound, as for q4k_gemm_f16).
 */
int q6k_gemm_f16(const void* w, int layout, int64_t rows, int64_t cols,
                 const uint16_t* hi, const uint16_t* lo, const uint16_t* bsum,
                 const float* inv_scale, int64_t tokens, float* y, void* stream);

/* q6k_gemm_blockdots - test export of the exact group dots of q6k_gemm:
 *   p : int32 [tokens][rows][cols/16], p[t][o][g] = P[t][o][g] above.
 * Bit-exact. */
int q6k_gemm_blockdots(const void* w, int layout, int64_t rows, int64_t cols,
                       const int8_t* q8, int64_t tokens, int32_t* p, void* stream);

/*
 * q4k_device_error - synchronise `stream` and read (then clear) the
 * library's device-side error word on the current device.  Returns Q4K_OK,
 * Q4K_ERR_DEVICE_TIMEOUT if a kernel abandoned a bounded wait since the last
 * read, or Q4K_ERR_CUDA if the synchronisation itself failed.
 */
int q4k_device_error(void* stream);

/*
 * q4k_selftest_wait_timeout - test export of the failure-detection path (no
 * counterpart on the pages): enqueues on `stream` a one-thread kernel whose
 * only wait is on a barrier that nothing completes.  The wait is bounded
 * like every wait in the library's kernels; after its limit (about two
 * seconds at the maximum SM clock) the kernel records a timeout in the
 * device error word and exits normally.  A following q4k_device_error()
 * then returns Q4K_ERR_DEVICE_TIMEOUT, and the context remains usable.
 */
int q4k_selftest_wait_timeout(void* stream);

/* Static, human-readable name of a status code. */
const char* q4k_status_string(int status);

/* Thread-local text of the last CUDA error seen by a call ("" if none). */
const char* q4k_last_error_string(void);

/* Library version, e.g. "q4k 0.1.0 sm_103a". */
const char* q4k_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q4K_H */
