/*
 * dualkv_layer.h -- C ABI of one decoder layer run on the packed layout.
 *
 * The DualKV repacking puts the micro-batch's N(P+R) tokens into P + NR rows
 * and runs the whole model on them, not only attention ("DualKV: Shared-Prompt
 * Flash Attention for Efficient RL Training with Large Rollouts and Long
 * Contexts"; arXiv abstract page: the data-pipeline redesign extends the token
 * reduction by rho = N(P+R)/(P+NR) "to the entire model"; forum page, "Two
 * changes", change 2).  That is exact because causal masking keeps every
 * prompt hidden state the same in all N sequences at every layer.  These
 * entry points run one pre-norm decoder layer of the Qwen3 family (the models
 * the pages train) on the packed rows, forward and backward, with the exact
 * shared-prompt attention of dualkv.h inside:
 *
 *     h1 = RMSNorm(x) * ln1
 *     q, k, v = split(h1 Wqkv^T);   q, k rotated by RoPE at the row positions
 *     a  = dualkv attention (groups as in dualkv_fwd_groups, scale 1/sqrt(d))
 *     x2 = x + a Wo^T
 *     h2 = RMSNorm(x2) * ln2
 *     y  = x2 + (silu(gate) * up) Wd^T,   [gate | up] = h2 Wgu^T
 *
 * (Qwen3's per-head q/k RMSNorm is left out: it acts on each row alone.)
 *
 * Positions: a prompt row sits at positions 0..P_g-1 of its group and a
 * response row continues its prompt: row j of a response is at P_g + j.
 * RMSNorm: r = 1/sqrt(mean(x^2) + eps).  RoPE: the feature pair (i, i + d/2)
 * of each head is rotated by pos * rope_base^(-2i/d).  silu(g) = g/(1+e^-g).
 *
 * Layouts (row-major, contiguous, device memory, 16-byte aligned):
 *   x, y, dy, dx : [T, hidden] bf16, T = sum over groups of P_g + sum R
 *   ln1, ln2     : [hidden] bf16
 *   wqkv         : [(Hq + 2*Hkv)*d, hidden] bf16 (q rows, then k rows, then v rows)
 *   wo           : [hidden, Hq*d] bf16
 *   wgu          : [2*inter, hidden] bf16 (gate rows, then up rows)
 *   wd           : [hidden, inter] bf16
 *   gradients    : the same shapes in fp32 (overwritten, not accumulated)
 * Accepted shapes: d in {64, 128}; Hq % Hkv == 0; Hq <= 4096; hidden % 8 == 0
 * and hidden <= 6144; inter % 8 == 0 and inter <= 2^24; the group rules of
 * dualkv_fwd_groups.
 *
 * Every step runs in this library's kernels on the caller's stream: the
 * GEMMs on the tcgen05 tensor cores (bf16 inputs, fp32 accumulation, bf16
 * activations and fp32 weight gradients), RMSNorm, RoPE, SwiGLU and the
 * attention.  The library allocates no device memory.
 *
 * Errors: the status codes of dualkv.h.  Arguments are checked before
 * anything is launched; a launch failure maps to DUALKV_ERR_CUDA, and a
 * bounded device wait that gives up is reported by dualkv_last_device_error().
 */
#ifndef DUALKV_LAYER_H_
#define DUALKV_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#include "dualkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t hidden;   /* model width */
  int32_t Hq, Hkv;  /* query / key-value heads */
  int32_t d;        /* head size, 64 or 128 */
  int32_t inter;    /* MLP width */
  float rope_base;  /* RoPE base (Qwen3: 1e6) */
  float eps;        /* RMSNorm epsilon (Qwen3: 1e-6) */
} dualkv_layer_config;

typedef struct {
  const void* ln1;
  const void* wqkv;
  const void* wo;
  const void* ln2;
  const void* wgu;
  const void* wd;
} dualkv_layer_weights;

typedef struct {
  float* ln1;
  float* wqkv;
  float* wo;
  float* ln2;
  float* wgu;
  float* wd;
} dualkv_layer_grads;

/*
 * Bytes of device workspace for one forward + backward of this shape: the
 * activations the forward saves for the backward and the backward's scratch.
 * Returns 0 for arguments the layer calls would reject.
 */
DUALKV_API size_t dualkv_layer_workspace_bytes(const dualkv_layer_config* cfg, int32_t G, const int64_t* P,
                                               const int32_t* N, const int32_t* R_lens);

/*
 * Forward: y = layer(x) on the packed rows of G groups (P, N, R_lens: host
 * arrays as in dualkv_fwd_groups).  workspace: at least
 * dualkv_layer_workspace_bytes() bytes, 256-byte aligned; the forward fills
 * it with the activations the backward reads.
 */
DUALKV_API int dualkv_layer_fwd(const dualkv_layer_config* cfg, const dualkv_layer_weights* w, const void* x,
                                int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens, void* y,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: given the forward's input x and dy (packed; a prompt row carries
 * the gradient of the one shared row, i.e. the sum over its group's
 * sequences), writes dx and the weight gradients.  workspace must hold what dualkv_layer_fwd saved for the
 * same x, weights and groups; the backward overwrites part of it, so each
 * forward serves one backward.
 */
DUALKV_API int dualkv_layer_bwd(const dualkv_layer_config* cfg, const dualkv_layer_weights* w, const void* x,
                                const void* dy, int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens, void* dx,
                                const dualkv_layer_grads* grads, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * Position ids of the packed rows (host): pos[t] for t < T, T = the packed row
 * count of the groups.  Returns DUALKV_OK, or DUALKV_ERR_INVALID_ARG for bad
 * groups or when T exceeds `capacity`.
 */
DUALKV_API int dualkv_packed_positions(int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens,
                                       int32_t* pos, int64_t capacity);

/*
 * One of the layer's GEMMs on its own (no counterpart on the DualKV pages;
 * exposed so that tests and benchmarks can check and time the tensor-core
 * GEMM the layer runs).  Row-major bf16 operands, fp32 accumulation:
 *   kind 0: Y[M,N] = A[M,K] . B[N,K]^T, bf16 Y; accumulate != 0 adds the
 *           result to what Y holds (Y = Y + A.B^T, one rounding);
 *   kind 1: Y[M,N] = A[M,K] . B[K,N], bf16 Y;
 *   kind 2: Y[M,N] = A[K,M]^T . B[K,N], fp32 Y (zeros when K == 0).
 * Every row length of A, B and Y (the contiguous dimension) must be a
 * multiple of 8, and every pointer 16-byte aligned.  M, N, K >= 0 and below
 * 2^31, M * N at most 2^40.  Returns DUALKV_OK, DUALKV_ERR_INVALID_ARG,
 * DUALKV_ERR_UNSUPPORTED (a row length not a multiple of 8, or M * N over
 * 2^40), DUALKV_ERR_ALIGNMENT or DUALKV_ERR_CUDA.
 */
DUALKV_API int dualkv_gemm(int32_t kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* Y,
                           int32_t accumulate, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DUALKV_LAYER_H_ */
