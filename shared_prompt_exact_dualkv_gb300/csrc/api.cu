// C ABI (include/dualkv.h): argument checks, the longest-first tile
// schedules, TMA tensor maps, workspace layout and the launch sequence.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/dualkv.h"
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace dkv {

__device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;

unsigned int* error_word_ptr() {
  static unsigned int* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

struct Shape {
  int64_t T = 0;
  int32_t P = 0, N = 0, Hq = 0, Hkv = 0, d = 0;
  std::vector<int32_t> R;
};

int check_shape(Shape* sh, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d) {
  if (N < 1 || N > kMaxSeq || R_lens == nullptr || P < 0 || Hq < 1 || Hkv < 1) return DUALKV_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DUALKV_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return DUALKV_ERR_UNSUPPORTED;
  int64_t T = P;
  sh->R.resize(N);
  for (int i = 0; i < N; ++i) {
    if (R_lens[i] < 0) return DUALKV_ERR_INVALID_ARG;
    sh->R[i] = R_lens[i];
    T += R_lens[i];
  }
  if (T >= (int64_t(1) << 31) || T * int64_t(Hq) * d >= (int64_t(1) << 40)) return DUALKV_ERR_INVALID_ARG;
  sh->T = T;
  sh->P = static_cast<int32_t>(P);
  sh->N = N;
  sh->Hq = Hq;
  sh->Hkv = Hkv;
  sh->d = d;
  return DUALKV_OK;
}

void fill_common(Sched* s, const Shape& sh, float scale) {
  s->T = static_cast<int32_t>(sh.T);
  s->P = sh.P;
  s->N = sh.N;
  s->Hq = sh.Hq;
  s->Hkv = sh.Hkv;
  s->group = sh.Hq / sh.Hkv;
  s->scale = scale;
  s->scale_log2 = scale * 1.4426950408889634f;
  s->off[0] = sh.P;
  for (int i = 0; i < sh.N; ++i) s->off[i + 1] = s->off[i] + sh.R[i];
  s->num_splits = 1;
  s->num_items = 0;
}

struct CostItem {
  int64_t cost;
  uint32_t item;
};

int finish_items(Sched* s, std::vector<CostItem>& v) {
  if (v.size() > static_cast<size_t>(kMaxItems)) return DUALKV_ERR_UNSUPPORTED;
  std::stable_sort(v.begin(), v.end(), [](const CostItem& a, const CostItem& b) { return a.cost > b.cost; });
  for (size_t i = 0; i < v.size(); ++i) s->items[i] = v[i].item;
  s->num_items = static_cast<int32_t>(v.size());
  return DUALKV_OK;
}

// Query-tile items (forward and dQ): cost = number of key tiles walked.
int build_query_sched(Sched* s, const Shape& sh, float scale) {
  fill_common(s, sh, scale);
  std::vector<CostItem> v;
  const int nP = ceil_div(sh.P, kTile);
  for (int t = 0; t < nP; ++t) v.push_back({t + 1, make_item(t, 0, 0)});
  for (int i = 0; i < sh.N; ++i) {
    const int nR = ceil_div(sh.R[i], kTile);
    for (int t = 0; t < nR; ++t) v.push_back({nP + t + 1, make_item(t, i + 1, 0)});
  }
  return finish_items(s, v);
}

// Sequence chunk boundaries of the prompt key tiles' work: split c covers
// responses [c*N/S, (c+1)*N/S); split 0 also takes the prompt's own queries.
int64_t prompt_item_cost(const Shape& sh, int j, int c, int S, const std::vector<int>& nR) {
  const int nP = ceil_div(sh.P, kTile);
  int64_t cost = (c == 0) ? (nP - j) : 0;
  for (int i = (c * sh.N) / S; i < ((c + 1) * sh.N) / S; ++i) cost += nR[i];
  return cost;
}

int auto_splits(const Shape& sh) {
  const int nP = ceil_div(sh.P, kTile);
  if (nP == 0) return 1;
  std::vector<int> nR(sh.N);
  int64_t resp_tiles = 0, total = 0;
  for (int i = 0; i < sh.N; ++i) {
    nR[i] = ceil_div(sh.R[i], kTile);
    resp_tiles += nR[i];
    total += int64_t(nR[i]) * (nR[i] + 1) / 2;  // response key tiles
  }
  total += int64_t(nP) * (nP + 1) / 2 + int64_t(nP) * resp_tiles;  // prompt key tiles
  total *= sh.Hkv;
  // Largest single item at most a quarter of one SM's fair share.
  const double target = std::max(1.0, double(total) / (4.0 * num_sms()));
  const double biggest = double(nP + resp_tiles);
  int S = static_cast<int>(std::ceil(biggest / target));
  S = std::max(1, std::min({S, sh.N, 16}));
  return S;
}

// Key-tile items (dK/dV): cost = number of query tiles walked per q-head.
int build_key_sched(Sched* s, const Shape& sh, float scale, int S) {
  fill_common(s, sh, scale);
  s->num_splits = S;
  std::vector<CostItem> v;
  std::vector<int> nR(sh.N);
  for (int i = 0; i < sh.N; ++i) nR[i] = ceil_div(sh.R[i], kTile);
  const int nP = ceil_div(sh.P, kTile);
  // Every (prompt key tile, split) is listed, even one whose sequence chunk
  // has no query tiles: in deterministic mode it must still write its
  // (zero) partial slice, which the fixed-order reduce reads.
  for (int j = 0; j < nP; ++j)
    for (int c = 0; c < S; ++c) v.push_back({prompt_item_cost(sh, j, c, S, nR), make_item(j, 0, c)});
  for (int i = 0; i < sh.N; ++i)
    for (int j = 0; j < nR[i]; ++j) v.push_back({nR[i] - j, make_item(j, i + 1, 0)});
  return finish_items(s, v);
}

int resolve_splits(const Shape& sh, int32_t num_splits) {
  if (num_splits <= 0) return auto_splits(sh);
  return std::max(1, std::min({num_splits, sh.N, 31}));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t D = 0, acc_k = 0, acc_v = 0, total = 0;
  size_t acc_floats = 0;  // floats in one of acc_k / acc_v
  size_t slice = 0;       // floats per split slice
  int S = 1;
};

WsLayout workspace_layout(const Shape& sh, int deterministic, int S) {
  WsLayout w;
  w.S = S;
  w.slice = size_t(sh.P) * sh.Hkv * sh.d;
  w.acc_floats = deterministic ? w.slice * S : w.slice;
  w.D = 0;
  w.acc_k = align256(size_t(sh.T) * sh.Hq * 4);
  w.acc_v = w.acc_k + align256(w.acc_floats * 4);
  w.total = w.acc_v + align256(w.acc_floats * 4);
  return w;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? DUALKV_OK : DUALKV_ERR_CUDA; }

// ------------------------------------------------------------------ tracing
constexpr int kTraceKernels = 5;

struct Trace {
  std::mutex mu;
  bool on = false;
  struct Rec {
    int kernel;
    cudaEvent_t a, b;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  double ms[kTraceKernels] = {};
  int64_t launches[kTraceKernels] = {};

  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
};

Trace& trace() {
  static Trace t;
  return t;
}

// Brackets one launch with events when tracing is on.
struct TraceScope {
  int kernel;
  cudaStream_t stream;
  cudaEvent_t a = nullptr, b = nullptr;
  TraceScope(int k, cudaStream_t s) : kernel(k), stream(s) {
    Trace& t = trace();
    std::lock_guard<std::mutex> lock(t.mu);
    if (!t.on) return;
    a = t.get();
    b = t.get();
    if (a) cudaEventRecord(a, stream);
  }
  ~TraceScope() {
    if (!a || !b) return;
    cudaEventRecord(b, stream);
    Trace& t = trace();
    std::lock_guard<std::mutex> lock(t.mu);
    t.pending.push_back({kernel, a, b});
  }
};

}  // namespace
}  // namespace dkv

using namespace dkv;

extern "C" {

int dualkv_version(void) { return 100; }

const char* dualkv_status_string(int status) {
  switch (status) {
    case DUALKV_OK: return "ok";
    case DUALKV_ERR_INVALID_ARG: return "invalid argument";
    case DUALKV_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128, Hq % Hkv == 0, tile count within limit)";
    case DUALKV_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case DUALKV_ERR_WORKSPACE: return "workspace missing or too small";
    case DUALKV_ERR_CUDA: return "CUDA runtime or launch error";
    case DUALKV_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int dualkv_fwd(const void* q, const void* k, const void* v, int64_t P, int32_t N, const int32_t* R_lens,
               int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale, void* out, float* lse, void* stream) {
  Shape sh;
  int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  if (!std::isfinite(softmax_scale)) return DUALKV_ERR_INVALID_ARG;
  if (sh.T == 0) return DUALKV_OK;
  if (!q || !k || !v || !out || !lse) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return DUALKV_ERR_ALIGNMENT;
  std::unique_ptr<Sched> s(new Sched);
  st = build_query_sched(s.get(), sh, softmax_scale);
  if (st != DUALKV_OK) return st;
  CUtensorMap mQ, mK, mV;
  if (!make_map_thd(&mQ, q, sh.T, Hq, d, kTile) || !make_map_thd(&mK, k, sh.T, Hkv, d, kTile) ||
      !make_map_thd(&mV, v, sh.T, Hkv, d, kTile))
    return DUALKV_ERR_CUDA;
  unsigned int* err = error_word_ptr();
  if (!err) return DUALKV_ERR_CUDA;
  TraceScope ts(0, static_cast<cudaStream_t>(stream));
  return map_cuda(launch_fwd(*s, d, mQ, mK, mV, out, lse, err, static_cast<cudaStream_t>(stream)));
}

size_t dualkv_bwd_workspace_bytes(int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv,
                                  int32_t d, int deterministic, int32_t num_splits) {
  Shape sh;
  if (check_shape(&sh, P, N, R_lens, Hq, Hkv, d) != DUALKV_OK) return 0;
  const int S = resolve_splits(sh, num_splits);
  return workspace_layout(sh, deterministic ? 1 : 0, S).total;
}

int dualkv_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
               int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d,
               float softmax_scale, int deterministic, int32_t num_splits, void* workspace,
               size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream) {
  Shape sh;
  int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  if (!std::isfinite(softmax_scale)) return DUALKV_ERR_INVALID_ARG;
  if (sh.T == 0) return DUALKV_OK;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return DUALKV_ERR_ALIGNMENT;
  const int det = deterministic ? 1 : 0;
  const int S = resolve_splits(sh, num_splits);
  const WsLayout ws = workspace_layout(sh, det, S);
  if (!workspace || workspace_bytes < ws.total) return DUALKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DUALKV_ERR_ALIGNMENT;

  std::unique_ptr<Sched> sq(new Sched), sk(new Sched);
  st = build_query_sched(sq.get(), sh, softmax_scale);
  if (st != DUALKV_OK) return st;
  st = build_key_sched(sk.get(), sh, softmax_scale, S);
  if (st != DUALKV_OK) return st;
  CUtensorMap mQ, mK, mV, mdO;
  if (!make_map_thd(&mQ, q, sh.T, Hq, d, kTile) || !make_map_thd(&mK, k, sh.T, Hkv, d, kTile) ||
      !make_map_thd(&mV, v, sh.T, Hkv, d, kTile) || !make_map_thd(&mdO, dout, sh.T, Hq, d, kTile))
    return DUALKV_ERR_CUDA;
  unsigned int* err = error_word_ptr();
  if (!err) return DUALKV_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* wb = static_cast<uint8_t*>(workspace);
  float* Dvec = reinterpret_cast<float*>(wb + ws.D);
  float* acc_k = reinterpret_cast<float*>(wb + ws.acc_k);
  float* acc_v = reinterpret_cast<float*>(wb + ws.acc_v);

  cudaError_t e;
  {
    TraceScope ts(1, cs);
    e = launch_preprocess(out, dout, Dvec, sh.T, Hq, d, det ? nullptr : acc_k,
                          det ? 0 : 2 * (ws.acc_v - ws.acc_k) / 4, cs);
  }
  if (e == cudaSuccess) {
    TraceScope ts(2, cs);
    e = launch_dkdv(*sk, d, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, det, err, cs);
  }
  if (e == cudaSuccess && sh.P > 0) {
    TraceScope ts(3, cs);
    e = launch_prompt_reduce(acc_k, acc_v, det ? S : 1, ws.slice, dk, dv, ws.slice, cs);
  }
  if (e == cudaSuccess) {
    TraceScope ts(4, cs);
    e = launch_dq(*sq, d, mQ, mK, mV, mdO, lse, Dvec, dq, err, cs);
  }
  return map_cuda(e);
}

int dualkv_trace_enable(int on) {
  Trace& t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  for (auto& r : t.pending) {
    cudaEventSynchronize(r.b);
    t.pool.push_back(r.a);
    t.pool.push_back(r.b);
  }
  t.pending.clear();
  for (int i = 0; i < kTraceKernels; ++i) {
    t.ms[i] = 0.0;
    t.launches[i] = 0;
  }
  t.on = on != 0;
  return DUALKV_OK;
}

int dualkv_trace_read(double* ms, int64_t* launches, int32_t n) {
  if ((!ms && !launches) || n < 0) return DUALKV_ERR_INVALID_ARG;
  Trace& t = trace();
  std::lock_guard<std::mutex> lock(t.mu);
  int status = DUALKV_OK;
  for (auto& r : t.pending) {
    float el = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&el, r.a, r.b) != cudaSuccess)
      status = DUALKV_ERR_CUDA;
    t.ms[r.kernel] += el;
    t.launches[r.kernel] += 1;
    t.pool.push_back(r.a);
    t.pool.push_back(r.b);
  }
  t.pending.clear();
  for (int i = 0; i < n && i < kTraceKernels; ++i) {
    if (ms) ms[i] = t.ms[i];
    if (launches) launches[i] = t.launches[i];
  }
  return status;
}

int dualkv_last_device_error(void* stream, int32_t* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DUALKV_ERR_CUDA;
  unsigned int w = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess) return DUALKV_ERR_CUDA;
  if (w == 0) return DUALKV_OK;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return DUALKV_ERR_CUDA;
  if (site) *site = static_cast<int32_t>(w >> 8);
  return static_cast<int>(w & 0xFFu) == DUALKV_ERR_TIMEOUT ? DUALKV_ERR_TIMEOUT : DUALKV_ERR_CUDA;
}

// ------------------------------------------------------------------ fixed scratch
// Backward pass for callers that cannot allocate: the workspace is this
// file-scope device array instead of caller memory.  In host code the name
// g_static_scratch is only a host-side stand-in for the symbol; its device
// address comes from cudaGetSymbolAddress, looked up once per device with
// that device current and cached.
static __device__ __align__(256) unsigned char g_static_scratch[DUALKV_STATIC_SCRATCH_BYTES];

static void* static_scratch_device_ptr() {
  static void* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess) return nullptr;
    cache[dev] = ptr;
  }
  return cache[dev];
}

int dualkv_bwd_static_workspace(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                const float* lse, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq,
                                int32_t Hkv, int32_t d, float softmax_scale, int deterministic, int32_t num_splits,
                                void* dq, void* dk, void* dv, void* stream) {
  Shape sh;
  const int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  if (sh.T == 0)
    return dualkv_bwd(q, k, v, out, dout, lse, P, N, R_lens, Hq, Hkv, d, softmax_scale, deterministic, num_splits,
                      nullptr, 0, dq, dk, dv, stream);
  const size_t need = dualkv_bwd_workspace_bytes(P, N, R_lens, Hq, Hkv, d, deterministic, num_splits);
  if (need > DUALKV_STATIC_SCRATCH_BYTES) return DUALKV_ERR_WORKSPACE;
  void* ws = static_scratch_device_ptr();
  if (!ws) return DUALKV_ERR_CUDA;
  return dualkv_bwd(q, k, v, out, dout, lse, P, N, R_lens, Hq, Hkv, d, softmax_scale, deterministic, num_splits,
                    ws, DUALKV_STATIC_SCRATCH_BYTES, dq, dk, dv, stream);
}

}  // extern "C"
