/*
 * dualkv.h -- C ABI of the GB300 (sm_103a) exact shared-prompt attention library.
 *
 * The operation ("DualKV: Shared-Prompt Flash Attention for Efficient RL
 * Training with Large Rollouts and Long Contexts"; research-map page, section
 * "Approach"; arXiv abstract page; forum page, "Two changes"): N response
 * sequences sampled from one P-token prompt are packed as P + sum_i R_i rows
 * -- the prompt once, then response 1 .. response N -- instead of N*(P+R)
 * replicated rows.  Attention on the packed rows is exactly the causal
 * attention of each replicated sequence [prompt ; response_i]:
 *   - a prompt row t attends to prompt keys 0..t;
 *   - a row of response i attends to every prompt key and, causally, to the
 *     keys of its own response up to and including itself.
 * The backward pass sums the prompt rows' dK/dV contributions of all N
 * sequences into the one packed copy.
 *
 * Conventions shared by every entry point
 *   T        = P + sum(R_lens)   packed rows; response i is rows [off_i, off_i + R_i)
 *            with off_0 = P, off_{i+1} = off_i + R_i.
 *   q, out, dout, dq : [T, Hq, d]  bf16, row-major, contiguous (device memory)
 *   k, v, dk, dv     : [T, Hkv, d] bf16, row-major, contiguous (device memory)
 *   lse              : [Hq, T] fp32 (device) -- natural log of
 *                      sum_j exp(softmax_scale * q . k_j) over the row's visible keys.
 *   R_lens           : HOST array of N int32 response lengths, read during the call.
 *   Grouped-query attention: q-head h reads kv-head h / (Hq / Hkv).
 *   Accepted shapes: d in {64, 128}; Hq % Hkv == 0; Hq <= 4096; 1 <= N <= 1024; P >= 0;
 *   R_i >= 0; T < 2^31; P and every R_i at most 8388480 rows (65535 tiles of
 *   128); every device pointer 16-byte aligned.  T == 0 is a no-op.  P == 0
 *   gives N independent causal sequences; N == 1 is one causal sequence of
 *   P + R_1 rows.  Work lists longer than one launch holds are split into
 *   several launches of the same kernel on `stream`.
 *   Packed dO of a prompt row is the gradient of the shared prompt row, i.e.
 *   the sum over the N replicated sequences of that row's gradient.
 *
 * Ownership: the caller owns every buffer, the workspace and the stream.  The
 * library allocates no device memory; the only state it keeps is a per-device
 * error word and a cached kernel configuration.  All work is enqueued on
 * `stream` (a cudaStream_t; NULL = legacy default stream) and the calls
 * return without synchronising.
 *
 * Errors: every entry point returns a dualkv_status.  Arguments are checked
 * before anything is launched; a rejected call launches nothing.  Launch
 * failures map to DUALKV_ERR_CUDA.  Device-side pipeline waits are bounded;
 * a wait that gives up records DUALKV_ERR_TIMEOUT in the device error word,
 * which dualkv_last_device_error() reports.
 */
#ifndef DUALKV_H_
#define DUALKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DUALKV_API __attribute__((visibility("default")))
#else
#define DUALKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DUALKV_OK = 0,
  DUALKV_ERR_INVALID_ARG = 1,  /* null pointer, negative length, N out of range, T mismatch */
  DUALKV_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, Hq % Hkv != 0, Hq > 4096, a segment over 65535 tiles */
  DUALKV_ERR_ALIGNMENT = 3,    /* a device pointer is not 16-byte aligned */
  DUALKV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than dualkv_bwd_workspace_bytes() */
  DUALKV_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
  DUALKV_ERR_TIMEOUT = 6,      /* a device-side wait gave up (reported by dualkv_last_device_error) */
  DUALKV_ERR_CHECK = 7         /* checks build only: a device-side index or pipeline check failed
                                  (reported by dualkv_last_device_error) */
} dualkv_status;

/*
 * Forward pass (research-map page, "Approach": one fused launch iterating over
 * the shared-context and per-sequence-response key regions).
 *   q, k, v       : device inputs, layouts above.
 *   P, N, R_lens  : packed layout; R_lens is a host array of N entries.
 *   softmax_scale : multiplies q . k before the softmax (usually 1/sqrt(d)).
 *   out           : device output [T, Hq, d] bf16 (written for all T rows).
 *   lse           : device output [Hq, T] fp32, natural-log LSE per row.
 *   stream        : cudaStream_t to enqueue on.
 * Returns DUALKV_OK or an error code; on error nothing is launched.
 */
DUALKV_API int dualkv_fwd(const void* q, const void* k, const void* v, int64_t P, int32_t N,
               const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale,
               void* out, float* lse, void* stream);

/*
 * Backward modes: the `deterministic` argument of the backward calls.
 *   DUALKV_BWD_ATOMIC (0): the prompt's dK/dV are summed over the sequences
 *     with fp32 atomics (research-map page, "Approach"); dQ comes from a
 *     separate kernel with one writer per row.
 *   DUALKV_BWD_DETERMINISTIC (1): per-split fp32 partials summed in a fixed
 *     order; bitwise reproducible.
 *   DUALKV_BWD_ATOMIC_FUSED_DQ (2): as mode 0, but dQ is computed in the
 *     dK/dV kernel, each key tile adding its share of dQ with fp32 atomics
 *     (no recomputation of S and dP); the workspace then also holds an fp32
 *     dQ accumulator of T*Hq*d*4 bytes, and dQ varies in the last bits from
 *     run to run.  On GB300 it is slower than mode 0 (the reductions stall
 *     the kernel); it is kept for comparison.
 */
#define DUALKV_BWD_ATOMIC 0
#define DUALKV_BWD_DETERMINISTIC 1
#define DUALKV_BWD_ATOMIC_FUSED_DQ 2

/*
 * Workspace bytes that dualkv_bwd needs for this shape and backward mode
 * (DUALKV_BWD_*).  num_splits is the number of sequence chunks a prompt key
 * tile's work is divided into (0 = library choice).  Returns 0 for arguments
 * dualkv_bwd would reject (including an unknown mode).
 */
DUALKV_API size_t dualkv_bwd_workspace_bytes(int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq,
                                  int32_t Hkv, int32_t d, int deterministic, int32_t num_splits);

/*
 * Backward pass (research-map page, "Approach": fused backward with the shared
 * prompt's gradients accumulated across the N sequences in fp32).
 *   q, k, v, out, lse : the forward's inputs and outputs (out and lse exactly
 *                       as dualkv_fwd wrote them).
 *   dout              : device [T, Hq, d] bf16 output gradient (prompt rows
 *                       carry the summed gradient of the shared rows).
 *   deterministic     : the backward mode, DUALKV_BWD_ATOMIC (0),
 *                       DUALKV_BWD_DETERMINISTIC (1, bitwise reproducible) or
 *                       DUALKV_BWD_ATOMIC_FUSED_DQ (2); other values are
 *                       DUALKV_ERR_INVALID_ARG.
 *   num_splits        : sequence chunks per prompt key tile (0 = library
 *                       choice; must match the value given to
 *                       dualkv_bwd_workspace_bytes).
 *   workspace         : device scratch of at least dualkv_bwd_workspace_bytes()
 *                       bytes, 256-byte aligned; contents need not be initialised.
 *   dq                : device output [T, Hq, d] bf16.
 *   dk, dv            : device outputs [T, Hkv, d] bf16.
 * Returns DUALKV_OK or an error code; on error nothing is launched.
 */
DUALKV_API int dualkv_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
               const float* lse, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq,
               int32_t Hkv, int32_t d, float softmax_scale, int deterministic, int32_t num_splits,
               void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream);

/*
 * Several prompt groups in one packed batch (research-map page, "Key
 * results": the speedups are quoted per micro-batch size, mb=8, without
 * saying whether it counts prompts or sequences; "Limitations": one shared
 * prefix per micro-batch group, no prefix trees).  These calls cover a
 * micro-batch that holds more than one prompt, each with its own responses.  The rows hold G groups one after another, group g
 * being its prompt of P[g] rows followed by its N[g] responses:
 *   rows = [prompt_0 ; resp_0,0 .. resp_0,N0-1 ; prompt_1 ; resp_1,0 .. ; ...]
 * and the visibility rule of the single-group calls holds inside each group
 * while no row sees any key of another group.  The result equals G separate
 * single-group calls on the groups' row ranges (with dualkv_bwd's reduction
 * mode and split count applied per group).
 *   G        : number of groups, >= 1.
 *   P        : HOST array of G prompt lengths (>= 0; 0 = the group's
 *              responses are plain causal sequences).
 *   N        : HOST array of G response counts (>= 0; 0 = a prompt alone).
 *   R_lens   : HOST array of sum(N) response lengths, group by group (may be
 *              NULL when sum(N) == 0).
 *   G + sum(N) must not exceed 1040.  Every other argument, layout, ownership
 *   rule and status code is that of the single-group call of the same name.
 */
DUALKV_API int dualkv_fwd_groups(const void* q, const void* k, const void* v, int32_t G, const int64_t* P,
                                 const int32_t* N, const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                 float softmax_scale, void* out, float* lse, void* stream);
DUALKV_API size_t dualkv_bwd_groups_workspace_bytes(int32_t G, const int64_t* P, const int32_t* N,
                                                    const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                                    int deterministic, int32_t num_splits);
DUALKV_API int dualkv_bwd_groups(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                 const float* lse, int32_t G, const int64_t* P, const int32_t* N,
                                 const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale,
                                 int deterministic, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                 void* dq, void* dk, void* dv, void* stream);

/*
 * One rank's part of a sequence-sharded step (research-map page, "Approach":
 * the shared prompt's gradients are accumulated across the N sequences in
 * fp32; "Key results" compares DualKV with sequence parallelism but the
 * pages describe no sharded DualKV).  When the N responses of a prompt are
 * spread over several ranks, every rank holds the whole prompt and its own
 * responses, packed as [prompt ; its responses], and these two calls let the
 * ranks divide the prompt's own causal attention instead of repeating it:
 * a rank takes the prompt query rows [prompt_row_lo, prompt_row_hi) and all
 * of its responses' query rows.  The responses need only the prompt's keys
 * and values, which every rank holds.
 *   prompt_row_lo, prompt_row_hi : 0 <= lo <= hi <= P; each a multiple of
 *                   128 or equal to P.  (0, P) takes the whole prompt, (P, P)
 *                   none of it.  Other values: DUALKV_ERR_INVALID_ARG.
 *
 * dualkv_fwd_partial: as dualkv_fwd, except that out and lse are written
 *   only for the prompt rows in [lo, hi) and for the response rows; the other
 *   prompt rows are left untouched (another rank computes them).
 *
 * dualkv_bwd_partial: as dualkv_bwd, except that
 *   - only the prompt query rows in [lo, hi) take part: the other prompt
 *     rows are treated as rows whose output gradient is zero, and their rows
 *     of dq (and dq_prompt) are left untouched.  dout, out and lse need to be
 *     valid only for the rows that take part;
 *   - the prompt rows' gradients are also returned unrounded, in fp32, when
 *     the pointers are not NULL (each may be NULL independently):
 *       dq_prompt : device [P, Hq, d] fp32, rows [lo, hi) written;
 *       dk_prompt, dv_prompt : device [P, Hkv, d] fp32, every prompt row
 *                   written with this call's sum over its query rows.
 *     Summing these over the ranks (in fp32) and rounding once gives the
 *     sharded step's prompt gradients; the bf16 prompt rows of dq/dk/dv hold
 *     this call's partial sums rounded to bf16.
 *   The workspace is sized by dualkv_bwd_workspace_bytes() for the same
 *   shape, mode and split count.  With (lo, hi) = (0, P) the bf16 outputs are
 *   those of dualkv_bwd.  Every fp32 pointer must be 16-byte aligned.
 */
DUALKV_API int dualkv_fwd_partial(const void* q, const void* k, const void* v, int64_t P, int32_t N,
                                  const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale,
                                  int64_t prompt_row_lo, int64_t prompt_row_hi, void* out, float* lse,
                                  void* stream);
DUALKV_API int dualkv_bwd_partial(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                  const float* lse, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq,
                                  int32_t Hkv, int32_t d, float softmax_scale, int deterministic,
                                  int32_t num_splits, int64_t prompt_row_lo, int64_t prompt_row_hi,
                                  void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv,
                                  float* dq_prompt, float* dk_prompt, float* dv_prompt, void* stream);

/*
 * Backward pass without any allocation (the DualKV pages have no counterpart;
 * this entry point exists for callers of this library, not for the method).
 * Some callers cannot call cudaMalloc or ask an allocator for memory at the
 * moment they run the backward pass: code running under a memory manager
 * that owns every byte of the device, code that must not synchronise (which
 * cudaMalloc/cudaFree can do), or plain-C hosts with no allocator at hand.
 * This variant takes the same arguments as dualkv_bwd minus the workspace
 * and uses instead a fixed scratch buffer of DUALKV_STATIC_SCRATCH_BYTES
 * (16 MiB) that lives inside the library as a device-global array; every
 * GPU that loads the library keeps those 16 MiB until the process exits.
 * The caller still owns and passes every input and output.
 *   - Shapes whose dualkv_bwd_workspace_bytes() exceeds 16 MiB are rejected
 *     with DUALKV_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the buffer's device address
 *     (with that device current); make that first call before any stream
 *     capture begins.
 *   - All calls share the one buffer and it keeps the last call's contents;
 *     the backward pass initialises every part of it that it reads, so no
 *     clearing is needed between calls.  Two calls whose kernels can run at
 *     the same time on the GPU (e.g. on unordered streams) race on the
 *     buffer and give wrong results: order them on one stream or with events.
 *   - It calls no cudaMalloc, cudaFree or allocating routine.
 * Returns the same status codes as dualkv_bwd.
 */
#define DUALKV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
DUALKV_API int dualkv_bwd_static_workspace(const void* q, const void* k, const void* v, const void* out,
                                           const void* dout, const float* lse, int64_t P, int32_t N,
                                           const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                           float softmax_scale, int deterministic, int32_t num_splits, void* dq,
                                           void* dk, void* dv, void* stream);

/*
 * Self-test of the failure detection (no counterpart on the DualKV pages).
 * Every pipeline wait in the kernels is bounded: a wait that does not
 * complete within its limit records DUALKV_ERR_TIMEOUT and the wait's site id
 * in the device error word, and the kernel returns instead of spinning.  This
 * call launches one thread that makes such a wait on an mbarrier phase that
 * nothing completes, with limit_ns (1 ns .. 10 s) and site (1 .. 2^24-1), so
 * that the path can be exercised without breaking a real pipeline.  After it,
 * dualkv_last_device_error() returns DUALKV_ERR_TIMEOUT and `site`.  Returns
 * DUALKV_OK, DUALKV_ERR_INVALID_ARG or DUALKV_ERR_CUDA.
 */
DUALKV_API int dualkv_selftest_wait_timeout(int64_t limit_ns, int32_t site, void* stream);

/* Static text for a dualkv_status value (never NULL). */
DUALKV_API const char* dualkv_status_string(int status);

/*
 * The CUDA code behind the calling thread's most recent DUALKV_ERR_CUDA from
 * any entry point of this library: a cudaError_t value, or, where a tensor
 * map was rejected, the driver's CUresult (-1 if the encoder could not be
 * reached).  0 if the thread has had no such failure.  Not reset by
 * successful calls.
 */
DUALKV_API int32_t dualkv_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns DUALKV_OK, DUALKV_ERR_TIMEOUT (a bounded device wait gave
 * up; *site, if non-NULL, receives the kernel-specific wait site id),
 * DUALKV_ERR_CHECK (checks build: a device-side check failed at *site) or
 * DUALKV_ERR_CUDA if the synchronisation itself failed.
 */
DUALKV_API int dualkv_last_device_error(void* stream, int32_t* site);

/*
 * Launch tracing (profiling aid).  dualkv_trace_enable(1) makes every later
 * dualkv_fwd / dualkv_bwd call in this process bracket each kernel it
 * launches with a pair of CUDA events recorded on the call's stream;
 * dualkv_trace_enable(0) stops that.  Enabling also clears the accumulated
 * totals.  dualkv_trace_read() synchronises on the recorded events and
 * returns, per kernel id, the summed device milliseconds and the launch
 * count since the last enable:
 *   0 forward, 1 backward preprocess (D = rowsum(dO*O)), 2 dK/dV,
 *   3 prompt dK/dV reduce + cast, 4 dQ.
 * `n` is the length of both arrays (at most 5 entries are written).
 * Events come from a pool owned by the library; no device memory is used.
 */
DUALKV_API int dualkv_trace_enable(int on);
DUALKV_API int dualkv_trace_read(double* ms, int64_t* launches, int32_t n);

/* Library version as major*10000 + minor*100 + patch. */
DUALKV_API int dualkv_version(void);

/*
 * 1 if this library is the checks build (compiled with DUALKV_CHECKS), else
 * 0.  No counterpart on the DualKV pages: a debugging aid.  In the checks
 * build every kernel tests, before each global access and each tile-copy
 * coordinate it computes, that the index lies inside its buffer, and at the
 * end of each CTA that its pipeline roles (copy producer, MMA issuer,
 * elementwise warps) completed the same number of steps as the schedule
 * gave them.  A failed check never traps: the access is skipped and the
 * first failure's site is recorded in the device error word, which
 * dualkv_last_device_error() returns as DUALKV_ERR_CHECK.  Results are those
 * of the regular build whenever no check fails.
 */
DUALKV_API int dualkv_checks_enabled(void);

#ifdef __cplusplus
}
#endif

#endif /* DUALKV_H_ */
