/*
 * muon.h -- C ABI of libmuon, the Muon optimizer step on whole weight matrices
 * for one GB300 GPU (sm_103a).
 *
 * The method: "Training a 1T-Parameter MoE on EU public infrastructure with
 * PyTorch and TorchTitan" (PyTorch blog), section "FlexShard: Muon without
 * communication".  Muon keeps one fp32 state per parameter and orthogonalises
 * each update with a few Newton-Schulz iterations that act on the whole
 * matrix; every rank owns complete expert matrices (hidden 6144, expert
 * hidden 1792 in the model-configuration table), so the step needs no
 * communication.  The page prints neither the iteration nor its constants;
 * this library takes them as arguments:
 *   momentum   buf <- mu*buf + g;  u <- g + mu*buf (Nesterov) or u <- buf
 *   orient     X = G^T when rows > cols (so X is m x n with m <= n)
 *   normalise  X <- X / (||X||_F + eps)
 *   iterate    A = X X^T;  B = b A + c A A;  X <- a X + B X     (steps times)
 *   update     W <- (1 - lr*wd) W - lr*scale*O
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device (or managed) memory on the
 *     current device.  The caller owns every buffer; the library keeps no
 *     per-call state and never frees caller memory.
 *   - All work is enqueued on `stream` (NULL = the legacy default stream) and
 *     returns without a host synchronisation.  Argument and launch errors are
 *     returned at once; device-side failures (a bounded wait that ran out)
 *     are reported by muon_get_device_status().
 *   - bf16 means IEEE bfloat16 (16-bit storage); conversions to bf16 round to
 *     nearest even.  Matrices are row-major, [batch][rows][cols], densely
 *     packed (matrix i starts at element i*rows*cols).
 *   - Calls return a muon_status (0 = success, negative = error).
 */
#ifndef MUON_H_
#define MUON_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t of the caller (same object); NULL is the legacy default stream. */
typedef struct CUstream_st *muon_stream_t;
/* A CUDA event (cudaEvent_t / CUevent), passed through unchanged. */
typedef struct CUevent_st *muon_event_t;

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = -1,  /* null pointer, negative size, bad coefficient pointer ... */
  MUON_ERR_UNSUPPORTED = -2,  /* shape, alignment or coefficients the tensor-core path does not take */
  MUON_ERR_CUDA = -3,         /* a CUDA runtime call or kernel launch failed */
  MUON_ERR_NO_MEMORY = -4,    /* workspace allocation failed or workspace too small */
  MUON_ERR_TIMEOUT = -5,      /* a device-side bounded wait ran out (kernel returned early) */
  MUON_ERR_DEVICE = -6        /* a device-side consistency check failed (non-finite input norm) */
} muon_status;

/* ---------------------------------------------------------------------------
 * Momentum (FlexShard section: one fp32 state per parameter).
 *   buf[i] <- fp32(fp32(mu*buf[i]) + g[i])
 *   u[i]   <- fp32(g[i] + fp32(mu*buf[i]))   if nesterov != 0 (new buf)
 *   u[i]   <- buf[i]                         otherwise
 * Each multiply and add is rounded to fp32 separately (no fused multiply-add),
 * so the result is bit-reproducible.
 *   grad       device, bf16, numel elements (read)
 *   momentum   device, fp32, numel elements (read and written in place)
 *   update_out device, bf16, numel elements (written; u rounded to bf16)
 *   numel >= 0; numel == 0 is a no-op.  Any alignment is accepted (16-byte
 *   aligned pointers take the vectorised path).
 * Errors: MUON_ERR_INVALID_ARG for null pointers with numel > 0 or numel < 0.
 */
int muon_momentum_update(const void *grad, float *momentum, void *update_out, int64_t numel,
                         float mu, int nesterov, muon_stream_t stream);

/* Same arithmetic with an fp32 gradient and an fp32 u (verification mode). */
int muon_momentum_update_f32(const float *grad, float *momentum, float *update_out, int64_t numel,
                             float mu, int nesterov, muon_stream_t stream);

/* ---------------------------------------------------------------------------
 * Batched Newton-Schulz orthogonalisation (FlexShard section: a few
 * Newton-Schulz iterations on the whole matrix, each matrix independent).
 *   X       device, bf16, [batch][m][n] row-major; read, and overwritten with
 *           the result in the same layout.  m > n is accepted: the iteration
 *           runs on X^T and the result is written back in X's layout.
 *   batch   >= 0 (0 is a no-op), m >= 1, n >= 1
 *   steps   0..1000 (0 = normalisation only)
 *   coeffs  host pointer to 3 floats (a, b, c); the quintic is
 *           (3.4445, -4.7750, 2.0315)
 *   eps     added to the Frobenius norm, eps >= 0 (1e-7 by convention)
 * Arithmetic: 16-bit operands on the tensor cores with fp32 accumulation,
 * fp32 epilogues, 16-bit storage (round to nearest even) of A and B, and X
 * carried between the steps as two halves (hi, and lo = bf16(X - hi)): the
 * tensor cores read hi, the a*X term uses hi + lo.  The 16-bit format is
 * bf16 when min(m, n) > 256; for smaller matrices it is fp16 scaled by
 * powers of two chosen from bounds that the coefficients give on every
 * iterate (8 times finer than bf16; the first step's B stays bf16), which
 * keeps small matrices, whose rounding errors average over few singular
 * directions, as accurate as large ones.  The 1/(||X||_F + eps) factor is
 * applied inside the first iteration's epilogues, not as a separate pass.
 * Requirements of the tensor-core path: m and n multiples of 8 and X 16-byte
 * aligned (TMA strides), else MUON_ERR_UNSUPPORTED; for min(m, n) <= 256
 * also coefficients under which no iterate's norm bound passes 2^54 (fp16
 * scaled by at least 2^-40), else MUON_ERR_UNSUPPORTED before any launch.
 * Workspace: muon_ns_batched allocates muon_ns_workspace_bytes() bytes
 * stream-ordered on `stream` (cudaMallocAsync/cudaFreeAsync from the device's
 * default memory pool); MUON_ERR_NO_MEMORY if that fails.
 * muon_ns_batched_ws uses caller memory instead (device, 256-byte aligned,
 * at least muon_ns_workspace_bytes(); it must not overlap X and must not be
 * used by other work until the enqueued work has finished).
 */
int muon_ns_batched(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3],
                    float eps, muon_stream_t stream);
size_t muon_ns_workspace_bytes(int64_t batch, int64_t m, int64_t n);
int muon_ns_batched_ws(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3],
                       float eps, void *workspace, size_t workspace_bytes, muon_stream_t stream);

/* Coefficient schedules (FlexShard section: "a few" Newton-Schulz iterations;
 * the page fixes neither their number nor their constants).  Step it uses
 * (a, b, c) = coeffs[3*it .. 3*it+2]; `coeffs` is a host array of 3*steps
 * floats (any non-null pointer when steps == 0).  Everything else as
 * muon_ns_batched / muon_ns_batched_f32, including the stream-ordered
 * workspace.  A schedule whose rows are all equal gives exactly the result of
 * the constant-coefficient call. */
int muon_ns_batched_schedule(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs,
                             float eps, muon_stream_t stream);
int muon_ns_batched_schedule_f32(float *X, int64_t batch, int64_t m, int64_t n, int steps, const float *coeffs,
                                 float eps, muon_stream_t stream);

/* ---------------------------------------------------------------------------
 * Newton-Schulz that allocates nothing.  Not part of the method itself: this
 * entry point exists for callers that cannot allocate device memory -- a host
 * that owns all device memory through its own arena and forbids allocations by
 * the libraries it loads, a runtime with a fixed memory budget that must not
 * allocate after start-up, or a plain C caller without a device allocator.
 * It computes exactly what muon_ns_batched computes (same kernels, same
 * arguments, same errors) on a scratch array of MUON_NS_STATIC_SCRATCH_BYTES
 * that the library reserves statically on the device.
 *   - Limit: muon_ns_workspace_bytes(batch, m, n) must not exceed
 *     MUON_NS_STATIC_SCRATCH_BYTES (96 MiB: one 1792 x 6144 expert matrix per
 *     call); larger calls return MUON_ERR_NO_MEMORY and touch nothing.
 *   - The scratch stays resident on every GPU that loads the library until
 *     the process exits.
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents (no part of it needs to start at zero).  Calls whose work
 *     overlaps on the GPU -- on different streams or from different host
 *     threads -- race on it: issue them on one stream.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define MUON_NS_STATIC_SCRATCH_BYTES (96ull << 20)
int muon_ns_batched_static(void *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3],
                           float eps, muon_stream_t stream);

/* fp32 verification mode: the same iteration in plain fp32 FFMA arithmetic
 * (no TF32, no bf16 rounding), any m, n >= 1; workspace allocated
 * stream-ordered like muon_ns_batched.  X is device fp32 [batch][m][n]. */
int muon_ns_batched_f32(float *X, int64_t batch, int64_t m, int64_t n, int steps, const float coeffs[3],
                        float eps, muon_stream_t stream);
size_t muon_ns_workspace_bytes_f32(int64_t batch, int64_t m, int64_t n);

/* ---------------------------------------------------------------------------
 * Parameter update with decoupled weight decay (the reading of the update the
 * page leaves open):
 *   W <- bf16(fp32(k_w*W) + fp32(k_o*O)),  k_w = fp32(1 - lr*wd),
 *   k_o = fp32(-lr*scale) (both constants formed in double on the host).
 *   param   device, bf16, [batch][rows][cols] (read and written in place)
 *   update  device, bf16, same layout (the orthogonalised O; read)
 *   scale   <= 0 selects sqrt(max(1, rows/cols)) on the stored shape
 * Errors: MUON_ERR_INVALID_ARG for null pointers or negative sizes.
 */
int muon_apply_update(void *param, const void *update, int64_t batch, int64_t rows, int64_t cols,
                      float lr, float weight_decay, float scale, muon_stream_t stream);

/* fp32 parameter and update, same formula without the bf16 rounding. */
int muon_apply_update_f32(float *param, const float *update, int64_t batch, int64_t rows, int64_t cols,
                          float lr, float weight_decay, float scale, muon_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole Muon step on matrices in device memory, fused (FlexShard section:
 * momentum, Newton-Schulz on each whole matrix and the update, with no
 * communication).  Computes, bit for bit, what
 *   muon_momentum_update(grad, momentum, u, batch*rows*cols, mu, nesterov, s);
 *   muon_ns_batched(u, batch, rows, cols, steps, coeffs, eps, s);
 *   muon_apply_update(param, u, batch, rows, cols, lr, weight_decay, scale, s);
 * compute, with no u array of the caller's and two passes over memory fewer:
 * the momentum kernel also sums the squares of u for the Frobenius norm, and
 * the last Newton-Schulz iteration applies the update to `param` in its
 * epilogue instead of storing O.
 *   param      device, bf16, [batch][rows][cols], read and written in place
 *   grad       device, bf16, same layout (read)
 *   momentum   device, fp32, same layout (read and written in place)
 *   steps, coeffs, eps   as muon_ns_batched;  lr, weight_decay, scale as
 *              muon_apply_update;  mu, nesterov as muon_momentum_update
 *   workspace  device, 256-byte aligned, at least
 *              muon_step_workspace_bytes(batch, rows, cols) bytes, used until
 *              the enqueued work has finished; NULL (with any workspace_bytes)
 *              allocates and frees it stream-ordered on `stream`
 * The four arrays must not overlap.  rows and cols must be multiples of 8 and
 * param, grad and momentum 16-byte aligned (else MUON_ERR_UNSUPPORTED).
 * Errors: MUON_ERR_INVALID_ARG as the three calls; MUON_ERR_NO_MEMORY for a
 * workspace smaller than required or a failed allocation.
 */
size_t muon_step_workspace_bytes(int64_t batch, int64_t rows, int64_t cols);
int muon_step_batched(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows, int64_t cols,
                      float mu, int nesterov, int steps, const float coeffs[3], float eps, float lr,
                      float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                      muon_stream_t stream);

/* The fused step with one (a, b, c) row per Newton-Schulz step: coeffs is a
 * host array of 3*steps floats as in muon_ns_batched_schedule (any non-null
 * pointer when steps == 0).  Bit for bit muon_momentum_update ->
 * muon_ns_batched_schedule -> muon_apply_update; everything else as
 * muon_step_batched. */
int muon_step_batched_schedule(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows,
                               int64_t cols, float mu, int nesterov, int steps, const float *coeffs, float eps,
                               float lr, float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                               muon_stream_t stream);

/* muon_step_batched whose one parameter-writing launch waits for an event.
 * Of the step's launches only the last (the final Newton-Schulz iteration
 * with the update, or the update alone when steps == 0) writes `param`; it is
 * ordered after `param_free` on `stream` (cudaStreamWaitEvent).  The momentum
 * and the earlier iterations are not, so work on other streams that still
 * reads the previous parameters (a copy to host memory, say) overlaps them.
 * param_free is an event the caller has recorded, or NULL (then this is
 * muon_step_batched).  Results are bit for bit those of muon_step_batched.
 * Errors as muon_step_batched, and MUON_ERR_CUDA if the wait cannot be
 * enqueued.
 */
int muon_step_batched_after(void *param, const void *grad, float *momentum, int64_t batch, int64_t rows,
                            int64_t cols, float mu, int nesterov, int steps, const float coeffs[3], float eps,
                            float lr, float weight_decay, float scale, void *workspace, size_t workspace_bytes,
                            muon_event_t param_free, muon_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole Muon step on matrices that live in host memory (FlexShard
 * section: with the parameters offloaded to host memory, Newton-Schulz runs on
 * the GPU).  param_host (bf16, in/out), grad_host (bf16) and momentum_host
 * (fp32, in/out) are page-locked host arrays (cudaHostAlloc /
 * cudaHostRegister) of batch matrices rows x cols.  The batch is streamed
 * through the GPU `chunk` matrices at a time (0: 8) in three device slots:
 * copies in and out run on two internal streams and overlap the compute of
 * the neighbouring chunk, which runs on `stream` and is muon_step_batched
 * (bit for bit muon_momentum_update -> muon_ns_batched ->
 * muon_apply_update).  The call returns once the work is enqueued; when
 * `stream` reaches it, the host arrays hold the updated parameters and
 * momentum (do not touch them before).
 * Device memory (3 slots of 12 bytes per element plus one step workspace
 * of `chunk` matrices) is allocated and freed stream-ordered on
 * `stream`.  Errors: MUON_ERR_INVALID_ARG for bad sizes or null pointers,
 * MUON_ERR_UNSUPPORTED for rows or cols not multiples of 8 or pageable host
 * memory, MUON_ERR_NO_MEMORY, MUON_ERR_CUDA.
 */
int muon_step_host(void *param_host, const void *grad_host, float *momentum_host, int64_t batch, int64_t rows,
                   int64_t cols, float mu, int nesterov, int steps, const float coeffs[3], float eps, float lr,
                   float weight_decay, float scale, int64_t chunk, muon_stream_t stream);

/* muon_step_host over several groups of matrices (each group one shape, its
 * own page-locked arrays and shape scale) in one pipeline: the chunks of all
 * groups, in order, rotate through the same device slots, so the host link
 * does not drain between groups as it does between separate calls (a model's
 * expert matrices come in several shapes).  Each group's result is bit for
 * bit that of muon_step_host on it.  Slots and workspace are sized for the
 * largest group shape.  A group with batch 0 is skipped.  Errors as
 * muon_step_host, checked for every group before anything is allocated or
 * enqueued, and MUON_ERR_INVALID_ARG for ngroups < 0 or groups == NULL with
 * ngroups > 0.
 */
typedef struct {
  void *param_host;          /* bf16, in/out */
  const void *grad_host;     /* bf16 */
  float *momentum_host;      /* fp32, in/out */
  int64_t batch, rows, cols;
  float scale;               /* <= 0: the default scale of rows x cols */
} muon_host_group;

int muon_step_host_grouped(const muon_host_group *groups, int ngroups, float mu, int nesterov, int steps,
                           const float coeffs[3], float eps, float lr, float weight_decay, int64_t chunk,
                           muon_stream_t stream);

/* ---------------------------------------------------------------------------
 * AdamW for the parameters Muon does not take (FlexShard section: routers and
 * embeddings use AdamW, with two fp32 states per parameter).  Reading taken:
 * decoupled weight decay with bias correction, every fp32 operation rounded
 * separately in this order (bit-reproducible):
 *   m <- (b1*m) + (c1*g);  v <- (b2*v) + (c2*(g*g));
 *   d <- sqrt(v / bc2) + eps;  W <- (kw*W) - (step_size*(m / d))
 * with c1 = 1-beta1, c2 = 1-beta2, bc2 = 1-beta2^step, step_size =
 * lr/(1-beta1^step), kw = 1-lr*weight_decay formed in double from the float
 * arguments and rounded once to fp32.
 *   param       device, bf16 (or fp32 for _f32), numel elements, in place
 *   grad        device, bf16 (fp32), numel elements
 *   exp_avg     device, fp32 first moment, in place;  exp_avg_sq: second moment
 *   step        >= 1, the 1-based step count the bias correction uses
 * Errors: MUON_ERR_INVALID_ARG for null pointers (numel > 0), numel < 0,
 * step < 1, betas outside [0, 1), negative eps or non-finite arguments.
 */
int muon_adamw_update(void *param, const void *grad, float *exp_avg, float *exp_avg_sq, int64_t numel, float lr,
                      float beta1, float beta2, float eps, float weight_decay, int64_t step, muon_stream_t stream);
int muon_adamw_update_f32(float *param, const float *grad, float *exp_avg, float *exp_avg_sq, int64_t numel,
                          float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                          muon_stream_t stream);

/* The default shape scale sqrt(max(1, rows/cols)). */
float muon_default_scale(int64_t rows, int64_t cols);

/* ---------------------------------------------------------------------------
 * Status, self-test and tracing helpers.
 */
/* Synchronises `stream`, then returns and clears the current device's error
 * word: MUON_ERR_TIMEOUT if a bounded wait ran out, MUON_ERR_DEVICE if a
 * Newton-Schulz input (or fused step's u) had a Frobenius norm that is not
 * finite in fp32 (an Inf or NaN entry, or entries beyond ~1.8e19; its output
 * is then zero or NaN), MUON_ERR_CUDA for a CUDA error, else MUON_OK. */
int muon_get_device_status(muon_stream_t stream);

/* Human-readable name of a muon_status value (static string). */
const char *muon_status_string(int status);

/* Upper bound, in nanoseconds, on every device-side wait of the tensor-core
 * kernels (default 2 s).  0 restores the default.  Returns the previous value. */
uint64_t muon_set_wait_timeout_ns(uint64_t timeout_ns);

/* Launches one kernel that waits on a barrier nothing will complete, with a
 * wait limit of timeout_ns, so that the timeout path can be checked: the
 * kernel gives up, records MUON_ERR_TIMEOUT in the error word and returns.
 * Returns the launch status; read the result with muon_get_device_status(). */
int muon_selftest_wait_timeout(uint64_t timeout_ns, muon_stream_t stream);

/* Number of kernels this library has launched in this process. */
int64_t muon_launch_count(void);

/* Fault injection on the host, for testing callers' error paths: the next
 * `count` device allocations the library makes for itself (the workspaces of
 * muon_ns_batched, muon_ns_batched_f32, the schedule variants and
 * muon_step_batched, and the slots of muon_step_host) fail as if the memory
 * pool were exhausted, without calling CUDA: the call returns
 * MUON_ERR_NO_MEMORY before it launches anything or touches its buffers.
 * count = 0 switches it off; count < 0 is MUON_ERR_INVALID_ARG.  Returns the
 * number of injected failures still pending before this call (>= 0).  Makes
 * no CUDA call. */
int muon_inject_alloc_failures(int count);

/* Tracing: between muon_trace_begin() and muon_trace_end(), every kernel
 * launch is bracketed by two CUDA events recorded on its own stream.
 * muon_trace_end() synchronises those events and fills up to max_entries
 * records (one per kernel kind that launched), returning how many kinds
 * launched (which may exceed max_entries) or a negative status. */
typedef struct {
  const char *kernel;     /* static name of the kernel kind */
  int64_t launches;       /* launches inside the traced region */
  double total_ms;        /* summed event-to-event duration */
} muon_trace_entry;

int muon_trace_begin(void);
int muon_trace_end(muon_trace_entry *entries, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* MUON_H_ */
