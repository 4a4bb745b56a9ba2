// C ABI of the packed decoder layer (include/dualkv_layer.h): argument
// checks, the workspace layout, and the launch sequence of the forward and
// backward passes.  Every step, GEMMs included (gemm.cu), runs in this
// library's kernels on the caller's stream.
#include <algorithm>
#include <cmath>
#include <memory>
#include <mutex>

#include "../../include/dualkv.h"
#include "../../include/dualkv_layer.h"
#include "kernels.h"
#include "layer_kernels.h"

namespace dkv {
namespace {

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Groups {
  int64_t T = 0;
  int64_t nres = 0;
};

// Checks the group arrays (the attention entry points check them again).
int check_groups(int32_t G, const int64_t* P, const int32_t* N, const int32_t* R, Groups* out) {
  if (G < 1 || G > kMaxSeg || !P || !N) return DUALKV_ERR_INVALID_ARG;
  int64_t T = 0, nres = 0;
  for (int g = 0; g < G; ++g) {
    if (P[g] < 0 || N[g] < 0) return DUALKV_ERR_INVALID_ARG;
    T += P[g];
    nres += N[g];
  }
  if (G + nres > kMaxSeg) return DUALKV_ERR_INVALID_ARG;
  if (nres > 0 && !R) return DUALKV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < nres; ++i) {
    if (R[i] < 0) return DUALKV_ERR_INVALID_ARG;
    T += R[i];
  }
  if (T >= (int64_t(1) << 31)) return DUALKV_ERR_INVALID_ARG;
  out->T = T;
  out->nres = nres;
  return DUALKV_OK;
}

int check_config(const dualkv_layer_config* c) {
  if (!c) return DUALKV_ERR_INVALID_ARG;
  if (c->hidden < 8 || c->Hq < 1 || c->Hkv < 1 || c->inter < 8) return DUALKV_ERR_INVALID_ARG;
  if (!(c->eps >= 0.f) || !std::isfinite(c->eps) || !(c->rope_base > 1.f) || !std::isfinite(c->rope_base))
    return DUALKV_ERR_INVALID_ARG;
  if (c->hidden % 8 || c->hidden > 6144 || c->inter % 8 || c->inter > (1 << 24) || c->Hq > 4096)
    return DUALKV_ERR_UNSUPPORTED;
  if ((c->d != 64 && c->d != 128) || c->Hq % c->Hkv) return DUALKV_ERR_UNSUPPORTED;
  return DUALKV_OK;
}

void fill_rowmap(RowMap* m, int32_t G, const int64_t* P, const int32_t* N, const int32_t* R) {
  int seg = 0, r = 0;
  int32_t row = 0;
  for (int g = 0; g < G; ++g) {
    m->off[seg] = row;
    m->pos0[seg] = 0;
    row += static_cast<int32_t>(P[g]);
    ++seg;
    for (int i = 0; i < N[g]; ++i, ++r, ++seg) {
      m->off[seg] = row;
      m->pos0[seg] = static_cast<int32_t>(P[g]);
      row += R[r];
    }
  }
  m->off[seg] = row;
  m->nseg = seg;
}

// Byte offsets of everything the layer keeps in the workspace.
struct LayerWs {
  // saved by the forward
  size_t h1, r1, q, k, v, a, lse, x2, r2, h2, gu, m;
  // forward transient, reused by the backward as dqkv
  size_t qkv;
  // backward scratch (dm reuses m; dgu is written over gu)
  size_t dh2, dx2, da, dq, dk, dv, dh1, part, attn;
  size_t attn_bytes, total;
};

LayerWs layout(const dualkv_layer_config& c, int64_t T, size_t attn_bytes) {
  LayerWs w{};
  const size_t H = c.hidden, I = c.inter, nq = size_t(c.Hq) * c.d, nk = size_t(c.Hkv) * c.d;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  w.h1 = take(T * H * 2);
  w.r1 = take(T * 4);
  w.q = take(T * nq * 2);
  w.k = take(T * nk * 2);
  w.v = take(T * nk * 2);
  w.a = take(T * nq * 2);
  w.lse = take(size_t(c.Hq) * T * 4);
  w.x2 = take(T * H * 2);
  w.r2 = take(T * 4);
  w.h2 = take(T * H * 2);
  w.gu = take(T * 2 * I * 2);
  w.m = take(T * I * 2);
  w.qkv = take(T * (nq + 2 * nk) * 2);
  w.dh2 = take(T * H * 2);
  w.dx2 = take(T * H * 2);
  w.da = take(T * nq * 2);
  w.dq = take(T * nq * 2);
  w.dk = take(T * nk * 2);
  w.dv = take(T * nk * 2);
  w.dh1 = take(T * H * 2);
  w.part = take(size_t(rmsnorm_bwd_blocks()) * H * 4);
  w.attn_bytes = attn_bytes;
  w.attn = take(std::max<size_t>(attn_bytes, 256));
  w.total = o;
  return w;
}

size_t attention_ws_bytes(const dualkv_layer_config& c, int32_t G, const int64_t* P, const int32_t* N,
                          const int32_t* R) {
  return dualkv_bwd_groups_workspace_bytes(G, P, N, R, c.Hq, c.Hkv, c.d, 0, 0);
}

// The layer's row-major GEMMs on the library's tensor-core kernels (gemm.cu),
// all on one stream; the first failure sticks.
struct Gemm {
  cudaStream_t stream = nullptr;
  unsigned int* err = nullptr;
  cudaError_t e = cudaSuccess;

  bool ok() const { return e == cudaSuccess; }
  int status() const { return ok() ? DUALKV_OK : cuda_fail(e); }
  // Y[rows, out] (+)= X[rows, in] . W[out, in]^T
  void xwT(int64_t rows, int out, int in, const void* X, const void* W, void* Y, float beta) {
    if (ok()) e = gemm_xwT(rows, out, in, X, W, Y, beta != 0.f, err, stream);
  }
  // dX[rows, in] = dY[rows, out] . W[out, in]
  void dyW(int64_t rows, int out, int in, const void* dY, const void* W, void* dX) {
    if (ok()) e = gemm_dyW(rows, in, out, dY, W, dX, err, stream);
  }
  // dW[out, in] (fp32) = dY[rows, out]^T . X[rows, in]
  void dW(int64_t rows, int out, int in, const void* dY, const void* X, float* dWp) {
    if (ok()) e = gemm_dW(out, in, rows, dY, X, dWp, err, stream);
  }
};

int begin_gemms(Gemm* g, cudaStream_t st) {
  g->stream = st;
  g->err = device_error_word();
  return g->err ? DUALKV_OK : cuda_fail(cudaGetLastError());
}

int weights_ok(const dualkv_layer_weights* w) {
  if (!w || !w->ln1 || !w->wqkv || !w->wo || !w->ln2 || !w->wgu || !w->wd) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(w->ln1) || !aligned16(w->wqkv) || !aligned16(w->wo) || !aligned16(w->ln2) || !aligned16(w->wgu) ||
      !aligned16(w->wd))
    return DUALKV_ERR_ALIGNMENT;
  return DUALKV_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DUALKV_OK : cuda_fail(e); }

}  // namespace
}  // namespace dkv

using namespace dkv;

extern "C" {

size_t dualkv_layer_workspace_bytes(const dualkv_layer_config* cfg, int32_t G, const int64_t* P, const int32_t* N,
                                    const int32_t* R_lens) {
  Groups gr;
  if (check_config(cfg) != DUALKV_OK || check_groups(G, P, N, R_lens, &gr) != DUALKV_OK) return 0;
  const size_t attn = attention_ws_bytes(*cfg, G, P, N, R_lens);
  if (attn == 0 && gr.T > 0) return 0;
  return layout(*cfg, gr.T, attn).total;
}

int dualkv_packed_positions(int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens, int32_t* pos,
                            int64_t capacity) {
  Groups gr;
  const int st = check_groups(G, P, N, R_lens, &gr);
  if (st != DUALKV_OK) return st;
  if (gr.T > capacity || (gr.T > 0 && !pos)) return DUALKV_ERR_INVALID_ARG;
  int64_t t = 0, r = 0;
  for (int g = 0; g < G; ++g) {
    for (int64_t j = 0; j < P[g]; ++j) pos[t++] = static_cast<int32_t>(j);
    for (int i = 0; i < N[g]; ++i, ++r)
      for (int32_t j = 0; j < R_lens[r]; ++j) pos[t++] = static_cast<int32_t>(P[g] + j);
  }
  return DUALKV_OK;
}

int dualkv_layer_fwd(const dualkv_layer_config* cfg, const dualkv_layer_weights* w, const void* x, int32_t G,
                     const int64_t* P, const int32_t* N, const int32_t* R_lens, void* y, void* workspace,
                     size_t workspace_bytes, void* stream) {
  int st = check_config(cfg);
  if (st != DUALKV_OK) return st;
  Groups gr;
  st = check_groups(G, P, N, R_lens, &gr);
  if (st != DUALKV_OK) return st;
  if (gr.T == 0) return DUALKV_OK;
  if ((st = weights_ok(w)) != DUALKV_OK) return st;
  if (!x || !y || !workspace) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return DUALKV_ERR_ALIGNMENT;
  const dualkv_layer_config& c = *cfg;
  const size_t attn = attention_ws_bytes(c, G, P, N, R_lens);
  if (attn == 0) return DUALKV_ERR_INVALID_ARG;
  const LayerWs L = layout(c, gr.T, attn);
  if (workspace_bytes < L.total) return DUALKV_ERR_WORKSPACE;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t T = gr.T;
  const int H = c.hidden, I = c.inter, nq = c.Hq * c.d, nk = c.Hkv * c.d;
  std::unique_ptr<RowMap> map(new RowMap);
  fill_rowmap(map.get(), G, P, N, R_lens);
  Gemm gm;
  if ((st = begin_gemms(&gm, cs)) != DUALKV_OK) return st;

  cudaError_t e = launch_rmsnorm_fwd(x, w->ln1, ws + L.h1, reinterpret_cast<float*>(ws + L.r1), T, H, c.eps, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  gm.xwT(T, nq + 2 * nk, H, ws + L.h1, w->wqkv, ws + L.qkv, 0.f);
  if (!gm.ok()) return gm.status();
  e = launch_rope_split(*map, ws + L.qkv, ws + L.q, ws + L.k, ws + L.v, static_cast<int>(T), c.Hq, c.Hkv, c.d,
                        c.rope_base, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  st = dualkv_fwd_groups(ws + L.q, ws + L.k, ws + L.v, G, P, N, R_lens, c.Hq, c.Hkv, c.d,
                         1.f / std::sqrt(static_cast<float>(c.d)), ws + L.a, reinterpret_cast<float*>(ws + L.lse),
                         stream);
  if (st != DUALKV_OK) return st;
  if ((e = cudaMemcpyAsync(ws + L.x2, x, size_t(T) * H * 2, cudaMemcpyDeviceToDevice, cs)) != cudaSuccess)
    return cuda_fail(e);
  gm.xwT(T, H, nq, ws + L.a, w->wo, ws + L.x2, 1.f);
  if (!gm.ok()) return gm.status();
  e = launch_rmsnorm_fwd(ws + L.x2, w->ln2, ws + L.h2, reinterpret_cast<float*>(ws + L.r2), T, H, c.eps, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  gm.xwT(T, 2 * I, H, ws + L.h2, w->wgu, ws + L.gu, 0.f);
  if (!gm.ok()) return gm.status();
  e = launch_swiglu_fwd(ws + L.gu, ws + L.m, T, I, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpyAsync(y, ws + L.x2, size_t(T) * H * 2, cudaMemcpyDeviceToDevice, cs)) != cudaSuccess)
    return cuda_fail(e);
  gm.xwT(T, H, I, ws + L.m, w->wd, y, 1.f);
  return gm.status();
}

int dualkv_layer_bwd(const dualkv_layer_config* cfg, const dualkv_layer_weights* w, const void* x, const void* dy,
                     int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens, void* dx,
                     const dualkv_layer_grads* grads, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_config(cfg);
  if (st != DUALKV_OK) return st;
  Groups gr;
  st = check_groups(G, P, N, R_lens, &gr);
  if (st != DUALKV_OK) return st;
  if ((st = weights_ok(w)) != DUALKV_OK) return st;
  if (!grads || !grads->ln1 || !grads->wqkv || !grads->wo || !grads->ln2 || !grads->wgu || !grads->wd)
    return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(grads->ln1) || !aligned16(grads->wqkv) || !aligned16(grads->wo) || !aligned16(grads->ln2) ||
      !aligned16(grads->wgu) || !aligned16(grads->wd))
    return DUALKV_ERR_ALIGNMENT;
  if (!workspace) return DUALKV_ERR_INVALID_ARG;
  if (gr.T > 0 && (!x || !dy || !dx)) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DUALKV_ERR_ALIGNMENT;
  const dualkv_layer_config& c = *cfg;
  const size_t attn = attention_ws_bytes(c, G, P, N, R_lens);
  if (attn == 0 && gr.T > 0) return DUALKV_ERR_INVALID_ARG;
  const LayerWs L = layout(c, gr.T, attn);
  if (workspace_bytes < L.total) return DUALKV_ERR_WORKSPACE;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t T = gr.T;
  const int H = c.hidden, I = c.inter, nq = c.Hq * c.d, nk = c.Hkv * c.d;
  std::unique_ptr<RowMap> map(new RowMap);
  fill_rowmap(map.get(), G, P, N, R_lens);
  Gemm gm;
  if ((st = begin_gemms(&gm, cs)) != DUALKV_OK) return st;

  // MLP: dWd, dm (over m), dgu (over gu), dWgu, dh2
  gm.dW(T, H, I, dy, ws + L.m, grads->wd);
  gm.dyW(T, H, I, dy, w->wd, ws + L.m);
  if (!gm.ok()) return gm.status();
  cudaError_t e = launch_swiglu_bwd(ws + L.gu, ws + L.m, ws + L.gu, T, I, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  gm.dW(T, 2 * I, H, ws + L.gu, ws + L.h2, grads->wgu);
  gm.dyW(T, 2 * I, H, ws + L.gu, w->wgu, ws + L.dh2);
  if (!gm.ok()) return gm.status();
  // second norm, with the residual path: dx2 = dy + RMSNorm'(dh2)
  e = launch_rmsnorm_bwd(ws + L.dh2, ws + L.x2, w->ln2, reinterpret_cast<const float*>(ws + L.r2), dy, ws + L.dx2,
                         reinterpret_cast<float*>(ws + L.part), grads->ln2, T, H, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  // attention output projection
  gm.dW(T, H, nq, ws + L.dx2, ws + L.a, grads->wo);
  gm.dyW(T, H, nq, ws + L.dx2, w->wo, ws + L.da);
  if (!gm.ok()) return gm.status();
  if (T > 0) {
    st = dualkv_bwd_groups(ws + L.q, ws + L.k, ws + L.v, ws + L.a, ws + L.da, reinterpret_cast<const float*>(ws + L.lse),
                           G, P, N, R_lens, c.Hq, c.Hkv, c.d, 1.f / std::sqrt(static_cast<float>(c.d)), 0, 0,
                           ws + L.attn, L.attn_bytes, ws + L.dq, ws + L.dk, ws + L.dv, stream);
    if (st != DUALKV_OK) return st;
  }
  e = launch_rope_merge(*map, ws + L.dq, ws + L.dk, ws + L.dv, ws + L.qkv, static_cast<int>(T), c.Hq, c.Hkv, c.d,
                        c.rope_base, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  gm.dW(T, nq + 2 * nk, H, ws + L.qkv, ws + L.h1, grads->wqkv);
  gm.dyW(T, nq + 2 * nk, H, ws + L.qkv, w->wqkv, ws + L.dh1);
  if (!gm.ok()) return gm.status();
  // first norm: dx = dx2 + RMSNorm'(dh1)
  e = launch_rmsnorm_bwd(ws + L.dh1, x, w->ln1, reinterpret_cast<const float*>(ws + L.r1), ws + L.dx2, dx,
                         reinterpret_cast<float*>(ws + L.part), grads->ln1, T, H, cs);
  return cuda_status(e);
}

int dualkv_gemm(int32_t kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* Y,
                int32_t accumulate, void* stream) {
  if (kind < 0 || kind > 2 || M < 0 || N < 0 || K < 0) return DUALKV_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim || K > lim) return DUALKV_ERR_INVALID_ARG;
  // tile counts are int: at most 2^40 output elements
  if (M * N > (int64_t(1) << 40)) return DUALKV_ERR_UNSUPPORTED;
  // row lengths of A, B and Y
  const int64_t la = kind == 2 ? M : K, lb = kind == 0 ? K : N;
  if (la % 8 || lb % 8 || N % 8) return DUALKV_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return DUALKV_OK;
  if (!Y || (K > 0 && (!A || !B))) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(Y)) return DUALKV_ERR_ALIGNMENT;
  unsigned int* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (kind == 0) {
    if (K == 0)
      return accumulate ? DUALKV_OK : cuda_status(cudaMemsetAsync(Y, 0, size_t(M) * N * 2, cs));
    e = gemm_xwT(M, static_cast<int>(N), static_cast<int>(K), A, B, Y, accumulate != 0, err, cs);
  } else if (kind == 1) {
    if (K == 0) return cuda_status(cudaMemsetAsync(Y, 0, size_t(M) * N * 2, cs));
    e = gemm_dyW(M, static_cast<int>(N), static_cast<int>(K), A, B, Y, err, cs);
  } else {
    e = gemm_dW(static_cast<int>(M), static_cast<int>(N), K, A, B, static_cast<float*>(Y), err, cs);
  }
  return cuda_status(e);
}

}  // extern "C"
