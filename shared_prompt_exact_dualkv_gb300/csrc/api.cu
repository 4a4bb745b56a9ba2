// C ABI (include/dualkv.h): argument checks, the tile schedules (longest
// first, each response's items together), TMA tensor maps, workspace layout
// and the launch sequence.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/dualkv.h"
#include "checks.cuh"
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

int l2_bytes() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 128 << 20;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return 128 << 20;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Packed batch shape: G prompt groups, group g = prompt of P[g] rows then
// N[g] responses (lengths in R, concatenated over groups).
struct Shape {
  int64_t T = 0;
  int32_t Hq = 0, Hkv = 0, d = 0;
  std::vector<int32_t> P, N, R;
  int64_t total_P = 0;
};

int check_dims(int32_t Hq, int32_t Hkv, int32_t d) {
  if (Hq < 1 || Hkv < 1) return DUALKV_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DUALKV_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return DUALKV_ERR_UNSUPPORTED;
  // a launch's grid is (work items) x (heads): at most 4096 x 4096 blocks
  if (Hq > 4096) return DUALKV_ERR_UNSUPPORTED;
  return DUALKV_OK;
}

int check_groups(Shape* sh, int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens, int32_t Hq,
                 int32_t Hkv, int32_t d) {
  if (G < 1 || G > kMaxSeg || !P || !N) return DUALKV_ERR_INVALID_ARG;
  int64_t nres = 0;
  for (int g = 0; g < G; ++g) {
    if (N[g] < 0 || P[g] < 0 || P[g] >= (int64_t(1) << 31)) return DUALKV_ERR_INVALID_ARG;
    nres += N[g];
  }
  if (G + nres > kMaxSeg) return DUALKV_ERR_INVALID_ARG;
  if (nres > 0 && !R_lens) return DUALKV_ERR_INVALID_ARG;
  const int st = check_dims(Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  sh->P.assign(G, 0);
  sh->N.assign(G, 0);
  sh->R.assign(static_cast<size_t>(nres), 0);
  int64_t T = 0, tp = 0;
  for (int g = 0; g < G; ++g) {
    sh->P[g] = static_cast<int32_t>(P[g]);
    sh->N[g] = N[g];
    T += P[g];
    tp += P[g];
  }
  // a segment's tile index has 16 bits in a work item
  constexpr int64_t kMaxSegRows = int64_t(0xFFFF) * kTile;
  for (int g = 0; g < G; ++g)
    if (P[g] > kMaxSegRows) return DUALKV_ERR_UNSUPPORTED;
  for (int64_t i = 0; i < nres; ++i) {
    if (R_lens[i] < 0) return DUALKV_ERR_INVALID_ARG;
    if (R_lens[i] > kMaxSegRows) return DUALKV_ERR_UNSUPPORTED;
    sh->R[i] = R_lens[i];
    T += R_lens[i];
  }
  if (T >= (int64_t(1) << 31)) return DUALKV_ERR_INVALID_ARG;
  sh->T = T;
  sh->total_P = tp;
  sh->Hq = Hq;
  sh->Hkv = Hkv;
  sh->d = d;
  return DUALKV_OK;
}

// One group of N responses (the original single-prompt interface).
int check_shape(Shape* sh, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d) {
  if (N < 1 || N > 1024 || R_lens == nullptr || P < 0) return DUALKV_ERR_INVALID_ARG;
  return check_groups(sh, 1, &P, &N, R_lens, Hq, Hkv, d);
}

// Segments in packed order, their group info and the prompt accumulator rows.
void fill_common(Sched* s, const Shape& sh, float scale) {
  s->T = static_cast<int32_t>(sh.T);
  s->Hq = sh.Hq;
  s->Hkv = sh.Hkv;
  s->group = sh.Hq / sh.Hkv;
  s->scale = scale;
  s->scale_log2 = scale * 1.4426950408889634f;
  s->num_splits = 1;
  s->num_items = 0;
  s->heads_outer = 0;
  s->pq_lo = 0;
  s->pq_hi = 0xFFFF;
  int seg = 0, r = 0;
  int32_t row = 0, acc = 0;
  for (size_t g = 0; g < sh.P.size(); ++g) {
    const int p = seg;
    s->off[seg] = row;
    s->info[seg] = p | (sh.N[g] << 16);
    s->acc_row[seg] = acc;
    row += sh.P[g];
    acc += sh.P[g];
    ++seg;
    for (int i = 0; i < sh.N[g]; ++i, ++r, ++seg) {
      s->off[seg] = row;
      s->info[seg] = p;
      s->acc_row[seg] = 0;
      row += sh.R[r];
    }
  }
  s->off[seg] = row;
  s->nseg = seg;
  s->acc_rows = acc;
}

// One work item with its cost (tiles walked) and its locality set: the
// items of one response segment read the same query (dK/dV) or key (forward,
// dQ) tiles of that response; every other item is a set of its own.
struct CostItem {
  int64_t cost;
  uint32_t item;
  int32_t locality;
};

// Longest-first by locality set: sets in order of their longest item, a
// set's items together, longest first.  The CTAs running at one time then
// come from one response and read its tiles at about the same time, so L2
// serves them once; listing items by cost alone interleaves all responses at
// each cost, and each response's tiles come back from HBM once per cost
// level.  Items in sets of their own keep the plain longest-first order.
std::vector<uint32_t> sorted_items(std::vector<CostItem>& v) {
  std::vector<int64_t> gmax;
  for (const CostItem& c : v) {
    if (c.locality >= static_cast<int32_t>(gmax.size())) gmax.resize(c.locality + 1, 0);
    gmax[c.locality] = std::max(gmax[c.locality], c.cost);
  }
  std::stable_sort(v.begin(), v.end(), [&](const CostItem& a, const CostItem& b) {
    if (gmax[a.locality] != gmax[b.locality]) return gmax[a.locality] > gmax[b.locality];
    if (a.locality != b.locality) return a.locality < b.locality;
    return a.cost > b.cost;
  });
  std::vector<uint32_t> out(v.size());
  for (size_t i = 0; i < v.size(); ++i) out[i] = v[i].item;
  return out;
}

// Block order of the query-tile kernels.  Every response query tile walks its
// prompt's keys and values; when those of all kv-heads exceed half of L2, the
// CTAs running together should share one kv-head's, so the heads become the
// outer block index.  Otherwise the items stay outer: the CTAs running
// together then come from fewer responses and share those responses' tiles.
int query_heads_outer(const Shape& sh) {
  const int64_t prompt_kv = int64_t(sh.total_P) * sh.Hkv * sh.d * 2 * 2;
  return prompt_kv > l2_bytes() / 2 ? 1 : 0;
}

// Query-tile items (forward and dQ): cost = number of key tiles walked.
// Prompt query tiles outside [pq_lo, pq_hi) are not listed.  The query tiles
// of one response form a locality set: they walk the same key tiles in the
// same order.
std::vector<uint32_t> query_items(const Sched& s) {
  std::vector<CostItem> v;
  int32_t nloc = 0;
  for (int seg = 0; seg < s.nseg; ++seg) {
    const int p = s.prompt_of(seg);
    const int nt = s.seg_tiles(seg);
    const int nA = (p == seg) ? 0 : s.seg_tiles(p);
    const int32_t g = nloc;
    if (p != seg && nt > 0) ++nloc;
    for (int t = 0; t < nt; ++t) {
      if (p == seg && (t < s.pq_lo || t >= s.pq_hi)) continue;
      v.push_back({nA + t + 1, make_item(t, seg, 0), p == seg ? nloc++ : g});
    }
  }
  return sorted_items(v);
}

// Sequence chunks of a prompt key tile's work: split c of group g covers its
// responses [c*N_g/S, (c+1)*N_g/S); split 0 also takes the prompt's own queries.
// Items are ordered group by group, longest first within each group: the
// CTAs running together then come from one group and walk the same query
// tiles, which L2 serves to all of them (ordering all groups' items by cost
// alone made a four-group batch's dK/dV 8% slower than four separate calls).
std::vector<uint32_t> key_items(const Sched& s, int S) {
  std::vector<uint32_t> out;
  std::vector<CostItem> v;
  int32_t nloc = 0;
  for (int seg = 0; seg < s.nseg; ++seg) {
    if (s.prompt_of(seg) == seg && !v.empty()) {  // a new group starts
      const std::vector<uint32_t> g = sorted_items(v);
      out.insert(out.end(), g.begin(), g.end());
      v.clear();
      nloc = 0;
    }
    const int nt = s.seg_tiles(seg);
    if (s.prompt_of(seg) == seg) {
      // Every (prompt key tile, split) is listed, even one whose sequence chunk
      // has no query tiles: in deterministic mode it must still write its
      // (zero) partial slice, which the fixed-order reduce reads.
      const int ng = s.responses_of(seg);
      for (int j = 0; j < nt; ++j)
        for (int c = 0; c < S; ++c) {
          // split 0 also walks the prompt's own query tiles j.. within [pq_lo, pq_hi)
          int64_t cost = (c == 0) ? std::max(0, std::min(nt, s.pq_hi) - std::max(j, s.pq_lo)) : 0;
          for (int i = seg + 1 + (c * ng) / S; i < seg + 1 + ((c + 1) * ng) / S; ++i) cost += s.seg_tiles(i);
          v.push_back({cost, make_item(j, seg, c), nloc++});
        }
    } else {
      // a response's key tiles read the same query tiles of that response
      for (int j = 0; j < nt; ++j) v.push_back({nt - j, make_item(j, seg, 0), nloc});
      ++nloc;
    }
  }
  const std::vector<uint32_t> g = sorted_items(v);
  out.insert(out.end(), g.begin(), g.end());
  return out;
}

int auto_splits(const Shape& sh) {
  int64_t total = 0, biggest = 0;
  int maxN = 1;
  size_t r = 0;
  for (size_t g = 0; g < sh.P.size(); ++g) {
    const int nP = ceil_div(sh.P[g], kTile);
    int64_t resp_tiles = 0;
    for (int i = 0; i < sh.N[g]; ++i, ++r) {
      const int nR = ceil_div(sh.R[r], kTile);
      resp_tiles += nR;
      total += int64_t(nR) * (nR + 1) / 2;
    }
    total += int64_t(nP) * (nP + 1) / 2 + int64_t(nP) * resp_tiles;
    if (nP > 0) biggest = std::max<int64_t>(biggest, nP + resp_tiles);
    maxN = std::max(maxN, sh.N[g]);
  }
  if (biggest == 0) return 1;
  total *= sh.Hkv;
  // Largest single item at most a quarter of one SM's fair share.
  const double target = std::max(1.0, double(total) / (4.0 * num_sms()));
  int S = static_cast<int>(std::ceil(double(biggest) / target));
  return std::max(1, std::min({S, maxN, 16}));
}

int resolve_splits(const Shape& sh, int32_t num_splits) {
  if (num_splits <= 0) return auto_splits(sh);
  int maxN = 1;
  for (int n : sh.N) maxN = std::max(maxN, n);
  return std::max(1, std::min({num_splits, maxN, 31}));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Backward modes (the `deterministic` argument of the ABI).
constexpr int kModeAtomic = DUALKV_BWD_ATOMIC;                // fp32 atomics for prompt dK/dV, separate dQ kernel
constexpr int kModeDeterministic = DUALKV_BWD_DETERMINISTIC;
constexpr int kModeFusedDq = DUALKV_BWD_ATOMIC_FUSED_DQ;      // fp32 atomics, dQ fused into the dK/dV kernel

bool mode_ok(int mode) { return mode == kModeAtomic || mode == kModeDeterministic || mode == kModeFusedDq; }

struct WsLayout {
  size_t D = 0, acc_k = 0, acc_v = 0, dq_acc = 0, total = 0;
  size_t acc_floats = 0;  // floats in one of acc_k / acc_v
  size_t slice = 0;       // floats per split slice
  int S = 1;
};

// D [Hq, T]; the prompt accumulators (one slice, or S in deterministic mode);
// in the fused mode the dQ accumulator [Hq][d/4][T][4] follows them, so that
// one zero-fill covers everything the atomics add into.
WsLayout workspace_layout(const Shape& sh, int mode, int S) {
  WsLayout w;
  w.S = S;
  w.slice = size_t(sh.total_P) * sh.Hkv * sh.d;
  w.acc_floats = mode == kModeDeterministic ? w.slice * S : w.slice;
  w.D = 0;
  w.acc_k = align256(size_t(sh.T) * sh.Hq * 4);
  w.acc_v = w.acc_k + align256(w.acc_floats * 4);
  w.dq_acc = w.acc_v + align256(w.acc_floats * 4);
  w.total = w.dq_acc + (mode == kModeFusedDq ? align256(size_t(sh.T) * sh.Hq * sh.d * 4) : 0);
  return w;
}

// Launches `launch` once per chunk of at most kMaxItems items.
template <typename F>
cudaError_t launch_chunks(Sched* s, const std::vector<uint32_t>& items, F&& launch) {
  for (size_t i0 = 0; i0 < items.size(); i0 += kMaxItems) {
    const size_t n = std::min(items.size() - i0, static_cast<size_t>(kMaxItems));
    std::copy(items.begin() + i0, items.begin() + i0 + n, s->items);
    s->num_items = static_cast<int32_t>(n);
    const cudaError_t e = launch(*s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? DUALKV_OK : cuda_fail(e); }

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

PromptMap* make_prompt_map(const Shape& sh) {
  PromptMap* m = new PromptMap;
  m->ngroups = 0;
  int64_t row = 0, acc = 0;
  size_t r = 0;
  for (size_t g = 0; g < sh.P.size(); ++g) {
    if (sh.P[g] > 0) {
      m->acc_row[m->ngroups] = static_cast<int32_t>(acc);
      m->packed_row[m->ngroups] = static_cast<int32_t>(row);
      ++m->ngroups;
    }
    row += sh.P[g];
    acc += sh.P[g];
    for (int i = 0; i < sh.N[g]; ++i, ++r) row += sh.R[r];
  }
  m->acc_row[m->ngroups] = static_cast<int32_t>(acc);
  return m;
}

// Prompt query tiles a call takes part in: [lo, hi) in tiles of kTile rows.
struct PromptPart {
  int32_t lo = 0, hi = 0xFFFF;
};

// Rows [row_lo, row_hi) of a prompt of P rows, tile-aligned (either end may be P).
int prompt_part(PromptPart* part, int64_t P, int64_t row_lo, int64_t row_hi) {
  if (row_lo < 0 || row_hi < row_lo || row_hi > P) return DUALKV_ERR_INVALID_ARG;
  if ((row_lo % kTile != 0 && row_lo != P) || (row_hi % kTile != 0 && row_hi != P)) return DUALKV_ERR_INVALID_ARG;
  part->lo = static_cast<int32_t>((row_lo + kTile - 1) / kTile);
  part->hi = static_cast<int32_t>((row_hi + kTile - 1) / kTile);
  return DUALKV_OK;
}

int fwd_impl(const Shape& sh, const void* q, const void* k, const void* v, float scale, void* out, float* lse,
             void* stream, PromptPart part = PromptPart()) {
  if (!std::isfinite(scale)) return DUALKV_ERR_INVALID_ARG;
  if (sh.T == 0) return DUALKV_OK;
  if (!q || !k || !v || !out || !lse) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return DUALKV_ERR_ALIGNMENT;
  std::unique_ptr<Sched> s(new Sched);
  fill_common(s.get(), sh, scale);
  s->pq_lo = part.lo;
  s->pq_hi = part.hi;
  s->heads_outer = query_heads_outer(sh);
  const std::vector<uint32_t> items = query_items(*s);
  CUtensorMap mQ, mK, mV;
  if (!make_map_thd(&mQ, q, sh.T, sh.Hq, sh.d, kTile) || !make_map_thd(&mK, k, sh.T, sh.Hkv, sh.d, kTile) ||
      !make_map_thd(&mV, v, sh.T, sh.Hkv, sh.d, kTile))
    return cuda_fail(last_map_result());
  unsigned int* err = error_word_ptr();
  if (!err) return cuda_fail(cudaGetLastError());
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return map_cuda(launch_chunks(s.get(), items, [&](const Sched& c) {
    TraceScope ts(0, cs);
    return launch_fwd(c, sh.d, mQ, mK, mV, out, lse, err, cs);
  }));
}

// fp32 copies of the prompt rows' gradients (accumulator row order), or nulls.
struct PromptF32 {
  float* dq = nullptr;
  float* dk = nullptr;
  float* dv = nullptr;
};

int bwd_impl(const Shape& sh, const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, float scale, int deterministic, int32_t num_splits, void* workspace,
             size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream, PromptPart part = PromptPart(),
             PromptF32 f32 = PromptF32()) {
  if (!std::isfinite(scale)) return DUALKV_ERR_INVALID_ARG;
  if (sh.T == 0) return DUALKV_OK;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return DUALKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(f32.dq) ||
      !aligned16(f32.dk) || !aligned16(f32.dv))
    return DUALKV_ERR_ALIGNMENT;
  const int mode = deterministic;
  if (!mode_ok(mode)) return DUALKV_ERR_INVALID_ARG;
  const int det = mode == kModeDeterministic ? 1 : 0;
  const bool fused = mode == kModeFusedDq;
  const int S = resolve_splits(sh, num_splits);
  const WsLayout ws = workspace_layout(sh, mode, S);
  if (!workspace || workspace_bytes < ws.total) return DUALKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DUALKV_ERR_ALIGNMENT;

  std::unique_ptr<Sched> sq(new Sched), sk(new Sched);
  fill_common(sq.get(), sh, scale);
  fill_common(sk.get(), sh, scale);
  sk->num_splits = S;
  sq->pq_lo = sk->pq_lo = part.lo;
  sq->pq_hi = sk->pq_hi = part.hi;
  sq->heads_outer = query_heads_outer(sh);
  const std::vector<uint32_t> q_items = query_items(*sq);
  const std::vector<uint32_t> k_items = key_items(*sk, S);
  std::unique_ptr<PromptMap> map(make_prompt_map(sh));
  CUtensorMap mQ, mK, mV, mdO;
  if (!make_map_thd(&mQ, q, sh.T, sh.Hq, sh.d, kTile) || !make_map_thd(&mK, k, sh.T, sh.Hkv, sh.d, kTile) ||
      !make_map_thd(&mV, v, sh.T, sh.Hkv, sh.d, kTile) || !make_map_thd(&mdO, dout, sh.T, sh.Hq, sh.d, kTile))
    return cuda_fail(last_map_result());
  unsigned int* err = error_word_ptr();
  if (!err) return cuda_fail(cudaGetLastError());
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* wb = static_cast<uint8_t*>(workspace);
  float* Dvec = reinterpret_cast<float*>(wb + ws.D);
  float* acc_k = reinterpret_cast<float*>(wb + ws.acc_k);
  float* acc_v = reinterpret_cast<float*>(wb + ws.acc_v);
  float* dq_acc = fused ? reinterpret_cast<float*>(wb + ws.dq_acc) : nullptr;

  cudaError_t e;
  {
    TraceScope ts(1, cs);
    // the atomic mode accumulates into acc_k/acc_v, which start at zero;
    // the deterministic mode overwrites every slice it reads
    e = launch_preprocess(out, dout, Dvec, sh.T, sh.Hq, sh.d, det ? nullptr : acc_k,
                          det ? 0 : (ws.total - ws.acc_k) / 4, cs);
  }
  if (e == cudaSuccess)
    e = launch_chunks(sk.get(), k_items, [&](const Sched& c) {
      TraceScope ts(2, cs);
      return launch_dkdv(c, sh.d, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, dq_acc, det, err, cs);
    });
  if (e == cudaSuccess && map->ngroups > 0) {
    TraceScope ts(3, cs);
    e = launch_prompt_reduce(acc_k, acc_v, det ? S : 1, ws.slice, dk, dv, f32.dk, f32.dv, *map, sh.Hkv * sh.d, err,
                             cs);
  }
  if (e == cudaSuccess && fused) {
    // dQ was summed in fp32 by the dK/dV kernel: scale and cast.  Prompt rows
    // outside the part this call takes are left untouched (a one-group call).
    TraceScope ts(4, cs);
    const bool one_prompt = sh.P.size() == 1;
    const int64_t pe = one_prompt ? sh.P[0] : 0;
    e = launch_dq_cast(dq_acc, dq, f32.dq, sh.T, sh.Hq, sh.d, scale, pe, int64_t(part.lo) * kTile,
                       std::min<int64_t>(int64_t(part.hi) * kTile, pe), cs);
  } else if (e == cudaSuccess) {
    e = launch_chunks(sq.get(), q_items, [&](const Sched& c) {
      TraceScope ts(4, cs);
      return launch_dq(c, sh.d, mQ, mK, mV, mdO, lse, Dvec, dq, f32.dq, err, cs);
    });
  }
  return map_cuda(e);
}

}  // namespace

unsigned int* device_error_word() { return error_word_ptr(); }

namespace {
thread_local int t_last_cuda_error = 0;
}

int cuda_fail(int code) {
  t_last_cuda_error = code;
  return DUALKV_ERR_CUDA;
}

int last_cuda_error() { return t_last_cuda_error; }

}  // namespace dkv

using namespace dkv;

extern "C" {

int dualkv_version(void) { return 100; }

int dualkv_checks_enabled(void) { return kChecks ? 1 : 0; }

const char* dualkv_status_string(int status) {
  switch (status) {
    case DUALKV_OK: return "ok";
    case DUALKV_ERR_INVALID_ARG: return "invalid argument";
    case DUALKV_ERR_UNSUPPORTED: return "unsupported shape (outside the accepted shapes the entry point documents)";
    case DUALKV_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case DUALKV_ERR_WORKSPACE: return "workspace missing or too small";
    case DUALKV_ERR_CUDA: return "CUDA runtime or launch error";
    case DUALKV_ERR_TIMEOUT: return "device-side wait timed out";
    case DUALKV_ERR_CHECK: return "device-side check failed (checks build)";
    default: return "unknown status";
  }
}

int dualkv_fwd(const void* q, const void* k, const void* v, int64_t P, int32_t N, const int32_t* R_lens,
               int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale, void* out, float* lse, void* stream) {
  Shape sh;
  const int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  return fwd_impl(sh, q, k, v, softmax_scale, out, lse, stream);
}

int dualkv_fwd_groups(const void* q, const void* k, const void* v, int32_t G, const int64_t* P, const int32_t* N,
                      const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale, void* out,
                      float* lse, void* stream) {
  Shape sh;
  const int st = check_groups(&sh, G, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  return fwd_impl(sh, q, k, v, softmax_scale, out, lse, stream);
}

size_t dualkv_bwd_workspace_bytes(int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv,
                                  int32_t d, int deterministic, int32_t num_splits) {
  Shape sh;
  if (check_shape(&sh, P, N, R_lens, Hq, Hkv, d) != DUALKV_OK || !mode_ok(deterministic)) return 0;
  return workspace_layout(sh, deterministic, resolve_splits(sh, num_splits)).total;
}

size_t dualkv_bwd_groups_workspace_bytes(int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens,
                                         int32_t Hq, int32_t Hkv, int32_t d, int deterministic,
                                         int32_t num_splits) {
  Shape sh;
  if (check_groups(&sh, G, P, N, R_lens, Hq, Hkv, d) != DUALKV_OK || !mode_ok(deterministic)) return 0;
  return workspace_layout(sh, deterministic, resolve_splits(sh, num_splits)).total;
}

int dualkv_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
               int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv, int32_t d,
               float softmax_scale, int deterministic, int32_t num_splits, void* workspace,
               size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream) {
  Shape sh;
  const int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  return bwd_impl(sh, q, k, v, out, dout, lse, softmax_scale, deterministic, num_splits, workspace,
                  workspace_bytes, dq, dk, dv, stream);
}

int dualkv_bwd_groups(const void* q, const void* k, const void* v, const void* out, const void* dout,
                      const float* lse, int32_t G, const int64_t* P, const int32_t* N, const int32_t* R_lens,
                      int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale, int deterministic,
                      int32_t num_splits, void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv,
                      void* stream) {
  Shape sh;
  const int st = check_groups(&sh, G, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  return bwd_impl(sh, q, k, v, out, dout, lse, softmax_scale, deterministic, num_splits, workspace,
                  workspace_bytes, dq, dk, dv, stream);
}

int dualkv_fwd_partial(const void* q, const void* k, const void* v, int64_t P, int32_t N, const int32_t* R_lens,
                       int32_t Hq, int32_t Hkv, int32_t d, float softmax_scale, int64_t prompt_row_lo,
                       int64_t prompt_row_hi, void* out, float* lse, void* stream) {
  Shape sh;
  int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  PromptPart part;
  st = prompt_part(&part, P, prompt_row_lo, prompt_row_hi);
  if (st != DUALKV_OK) return st;
  return fwd_impl(sh, q, k, v, softmax_scale, out, lse, stream, part);
}

int dualkv_bwd_partial(const void* q, const void* k, const void* v, const void* out, const void* dout,
                       const float* lse, int64_t P, int32_t N, const int32_t* R_lens, int32_t Hq, int32_t Hkv,
                       int32_t d, float softmax_scale, int deterministic, int32_t num_splits, int64_t prompt_row_lo,
                       int64_t prompt_row_hi, void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv,
                       float* dq_prompt, float* dk_prompt, float* dv_prompt, void* stream) {
  Shape sh;
  int st = check_shape(&sh, P, N, R_lens, Hq, Hkv, d);
  if (st != DUALKV_OK) return st;
  PromptPart part;
  st = prompt_part(&part, P, prompt_row_lo, prompt_row_hi);
  if (st != DUALKV_OK) return st;
  PromptF32 f32;
  f32.dq = dq_prompt;
  f32.dk = dk_prompt;
  f32.dv = dv_prompt;
  return bwd_impl(sh, q, k, v, out, dout, lse, softmax_scale, deterministic, num_splits, workspace,
                  workspace_bytes, dq, dk, dv, stream, part, f32);
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
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&el, r.a, r.b);
    if (e != cudaSuccess) status = cuda_fail(e);
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

int32_t dualkv_last_cuda_error(void) { return last_cuda_error(); }

int dualkv_selftest_wait_timeout(int64_t limit_ns, int32_t site, void* stream) {
  if (limit_ns < 1 || limit_ns > 10000000000ll || site < 1 || site > 0xFFFFFF) return DUALKV_ERR_INVALID_ARG;
  unsigned int* err = error_word_ptr();
  if (!err) return cuda_fail(cudaGetLastError());
  return map_cuda(launch_wait_timeout_selftest(err, static_cast<uint64_t>(limit_ns), static_cast<uint32_t>(site),
                                               static_cast<cudaStream_t>(stream)));
}

int dualkv_last_device_error(void* stream, int32_t* site) {
  if (site) *site = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int w = 0;
  if ((e = cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w))) != cudaSuccess) return cuda_fail(e);
  if (w == 0) return DUALKV_OK;
  const unsigned int zero = 0;
  if ((e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero))) != cudaSuccess) return cuda_fail(e);
  if (site) *site = static_cast<int32_t>(w >> 8);
  const int kind = static_cast<int>(w & 0xFFu);
  return (kind == DUALKV_ERR_TIMEOUT || kind == DUALKV_ERR_CHECK) ? kind : DUALKV_ERR_CUDA;
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
  if (!ws) return cuda_fail(cudaGetLastError());
  return dualkv_bwd(q, k, v, out, dout, lse, P, N, R_lens, Hq, Hkv, d, softmax_scale, deterministic, num_splits,
                    ws, DUALKV_STATIC_SCRATCH_BYTES, dq, dk, dv, stream);
}

}  // extern "C"
