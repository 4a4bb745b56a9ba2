// Host-side launchers of the per-token kernels of the packed decoder layer.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace dkv {

// Segments of the packed rows and the position of each segment's first row:
// row t of segment s (off[s] <= t < off[s+1]) sits at position pos0[s] + t - off[s].
struct RowMap {
  int32_t nseg;
  int32_t off[kMaxSeg + 1];
  int32_t pos0[kMaxSeg];
};

// y = x * r * w per row, r = 1/sqrt(mean(x^2) + eps) saved to rstd [rows].
// x, y [rows, hidden] bf16, w [hidden] bf16; hidden % 8 == 0, hidden <= 6144.
cudaError_t launch_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t rows, int hidden,
                               float eps, cudaStream_t st);

// dx = dres + RMSNorm'(dy) (row-parallel kernel); dw [hidden] fp32 = sum over
// rows of dy*x*r (per-chunk partials, then a fixed-order column sum).  part is
// fp32 scratch of rmsnorm_bwd_blocks() * hidden floats.
cudaError_t launch_rmsnorm_bwd(const void* dy, const void* x, const void* w, const float* rstd, const void* dres,
                               void* dx, float* part, float* dw, int64_t rows, int hidden, cudaStream_t st);
int rmsnorm_bwd_blocks();

// qkv [T, (Hq+2Hkv)*d] -> q [T,Hq,d], k [T,Hkv,d] rotated at the rows'
// positions, v [T,Hkv,d] copied.  d in {64, 128}.
cudaError_t launch_rope_split(const RowMap& map, const void* qkv, void* q, void* k, void* v, int T, int Hq, int Hkv,
                              int d, double rope_base, cudaStream_t st);

// The transpose: dq, dk rotated back and dv -> dqkv [T, (Hq+2Hkv)*d].
cudaError_t launch_rope_merge(const RowMap& map, const void* dq, const void* dk, const void* dv, void* dqkv, int T,
                              int Hq, int Hkv, int d, double rope_base, cudaStream_t st);

// m [rows, inter] = silu(gate) * up, gu [rows, 2*inter] = [gate | up]; inter % 8 == 0.
cudaError_t launch_swiglu_fwd(const void* gu, void* m, int64_t rows, int inter, cudaStream_t st);

// dgu = [dgate | dup] from dm and gu (dgu may be gu itself).
cudaError_t launch_swiglu_bwd(const void* gu, const void* dm, void* dgu, int64_t rows, int inter, cudaStream_t st);

// bf16 GEMMs on the tensor cores (gemm.cu); row-major operands, fp32
// accumulation.  Every column count and K must be a multiple of 8.
//   gemm_xwT: Y[M,N] = X[M,K] . W[N,K]^T (+ Y when accumulate), bf16 out.
//   gemm_dyW: dX[M,N] = dY[M,K] . W[K,N], bf16 out.
//   gemm_dW:  dW[M,N] = dY[K,M]^T . X[K,N], fp32 out (zero when K == 0).
// `err` is the device error word (bounded pipeline waits record timeouts).
cudaError_t gemm_xwT(int64_t M, int N, int K, const void* X, const void* W, void* Y, bool accumulate,
                     unsigned int* err, cudaStream_t stream);
cudaError_t gemm_dyW(int64_t M, int N, int K, const void* dY, const void* W, void* dX, unsigned int* err,
                     cudaStream_t stream);
cudaError_t gemm_dW(int M, int N, int64_t K, const void* dY, const void* X, float* dW, unsigned int* err,
                    cudaStream_t stream);

}  // namespace dkv
