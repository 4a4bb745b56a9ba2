// Per-token kernels of the packed decoder layer: RMSNorm (forward, backward
// and its weight-gradient reduction), RoPE at the packed positions (fused with
// the q/k/v split and, backward, the merge), and the SwiGLU activation.
//
// The DualKV pages (arXiv abstract page; forum page, "Two changes", change 2)
// point out that causal masking keeps every prompt hidden state the same in
// all N sequences, so every per-token operation of the model runs once on the
// P + NR packed rows.  The only per-token operation that must know where a row
// sits in its sequence is RoPE: a response row continues its prompt, so its
// position is P_g + (row - response start).
#include <cuda_bf16.h>

#include "layer_kernels.h"

namespace dkv {
namespace {

constexpr int kNormThreads = 128;  // 4 warps, one row per warp at a time

__device__ __forceinline__ void unpack8(uint4 v, float* f) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&t);
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Lane l of a warp owns the 8-column groups l, l + 32, l + 64, ... of a row.
template <int NG>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_fwd_kernel(const uint4* __restrict__ x,
                                                                  const uint4* __restrict__ w, uint4* __restrict__ y,
                                                                  float* __restrict__ rstd, int64_t rows, int groups,
                                                                  float eps) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t(blockIdx.x) * kNormThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kNormThreads) >> 5;
  const float inv_h = 1.f / (8.f * groups);
  for (int64_t r = warp0; r < rows; r += nwarps) {
    uint4 pk[NG];  // the row stays packed (bf16) between the two passes
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int gi = lane + 32 * j;
      if (gi < groups) {
        float v[8];
        pk[j] = x[r * groups + gi];
        unpack8(pk[j], v);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
      }
    }
    ss = warp_sum(ss);
    const float rs = rsqrtf(ss * inv_h + eps);
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int gi = lane + 32 * j;
      if (gi < groups) {
        float v[8], wf[8], o[8];
        unpack8(pk[j], v);
        unpack8(w[gi], wf);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = v[e] * rs * wf[e];
        y[r * groups + gi] = pack8(o);
      }
    }
    if (lane == 0) rstd[r] = rs;
  }
}

// dx = dres + r*(w*dy) - (r^3/H) * x * sum(w*dy*x), one warp per row; the
// second pass reads the row again (from L1).
template <int NG>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_dx_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ x, const uint4* __restrict__ w,
    const float* __restrict__ rstd, const uint4* __restrict__ dres, uint4* __restrict__ dx, int64_t rows,
    int groups) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t(blockIdx.x) * kNormThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kNormThreads) >> 5;
  const float inv_h = 1.f / (8.f * groups);
  for (int64_t r = warp0; r < rows; r += nwarps) {
    float dot = 0.f;
    const float rs = rstd[r];
#pragma unroll 4
    for (int j = 0; j < NG; ++j) {
      const int gi = lane + 32 * j;
      if (gi < groups) {
        float g[8], xv[8], wf[8];
        unpack8(dy[r * groups + gi], g);
        unpack8(x[r * groups + gi], xv);
        unpack8(w[gi], wf);
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(g[e] * wf[e], xv[e], dot);
      }
    }
    dot = warp_sum(dot);
    const float c = rs * rs * rs * dot * inv_h;
#pragma unroll 4
    for (int j = 0; j < NG; ++j) {
      const int gi = lane + 32 * j;
      if (gi < groups) {
        float g[8], xv[8], wf[8], d0[8], o[8];
        unpack8(dy[r * groups + gi], g);
        unpack8(x[r * groups + gi], xv);
        unpack8(w[gi], wf);
        unpack8(dres[r * groups + gi], d0);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = d0[e] + rs * (g[e] * wf[e]) - c * xv[e];
        dx[r * groups + gi] = pack8(o);
      }
    }
  }
}

// Partial dw of a contiguous chunk of rows: thread t of the block owns the 8
// columns of group t (and t + blockDim, ...) and sums dy*x*r over the chunk;
// part[blockIdx.x][column] = that sum.
__global__ void __launch_bounds__(256) rmsnorm_dw_kernel(const uint4* __restrict__ dy, const uint4* __restrict__ x,
                                                         const float* __restrict__ rstd, float* __restrict__ part,
                                                         int64_t rows, int groups) {
  const int64_t chunk = (rows + gridDim.x - 1) / gridDim.x;
  const int64_t r0 = int64_t(blockIdx.x) * chunk;
  const int64_t r1 = r0 + chunk < rows ? r0 + chunk : rows;
  for (int gi = threadIdx.x; gi < groups; gi += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int64_t r = r0; r < r1; ++r) {
      float g[8], xv[8];
      unpack8(dy[r * groups + gi], g);
      unpack8(x[r * groups + gi], xv);
      const float rs = rstd[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(g[e] * xv[e], rs, acc[e]);
    }
    float4* dst = reinterpret_cast<float4*>(part + int64_t(blockIdx.x) * groups * 8 + gi * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// dw[c] = sum over the blocks' partials, in block order.
__global__ void __launch_bounds__(256) column_sum_kernel(const float* __restrict__ part, float* __restrict__ dw,
                                                         int nblocks, int H) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  float s = 0.f;
  for (int b = 0; b < nblocks; ++b) s += part[int64_t(b) * H + c];
  dw[c] = s;
}

// Position of packed row t: rows [off[s], off[s+1]) of segment s sit at
// positions pos0[s] + (t - off[s]).
__device__ __forceinline__ int32_t row_position(const RowMap& m, int32_t t) {
  int lo = 0, hi = m.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m.off[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return m.pos0[lo] + (t - m.off[lo]);
}

// One block per row (grid-stride).  Forward: qkv [T, (Hq+2Hkv)*d] -> q, k
// rotated, v copied.  Backward (BWD): dq, dk rotated back, dv copied -> dqkv.
// The angle pos * base^(-2i/d) is formed and reduced modulo 2*pi in fp64, so
// the fp32 sine and cosine are accurate to fp32 rounding at any position.
template <int D, bool BWD>
__global__ void __launch_bounds__(128) rope_kernel(const __grid_constant__ RowMap map, const uint4* __restrict__ src,
                                                   const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                                                   uint4* __restrict__ dst, uint4* __restrict__ dst_k,
                                                   uint4* __restrict__ dst_v, int T, int Hq, int Hkv,
                                                   double log2_base) {
  constexpr int kHalf = D / 2;
  constexpr int kG = kHalf / 8;  // 8-element groups per half head
  __shared__ double inv_freq[kHalf];
  __shared__ float cs[kHalf], sn[kHalf];
  for (int i = threadIdx.x; i < kHalf; i += blockDim.x) inv_freq[i] = exp2(-2.0 * i / D * log2_base);
  const int W = (Hq + 2 * Hkv) * D / 8;  // uint4 per packed qkv row
  const double two_pi = 6.283185307179586476925286766559;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();  // previous row's readers are done with cs/sn
    const int32_t pos = row_position(map, t);
    for (int i = threadIdx.x; i < kHalf; i += blockDim.x) {
      const double a = remainder(static_cast<double>(pos) * inv_freq[i], two_pi);
      float s, c;
      sincosf(static_cast<float>(a), &s, &c);
      cs[i] = c;
      sn[i] = BWD ? -s : s;
    }
    __syncthreads();
    const int nrot = (Hq + Hkv) * kG;
    for (int u = threadIdx.x; u < nrot; u += blockDim.x) {
      const int head = u / kG;  // q heads first, then k heads
      const int g = u % kG;
      const bool is_q = head < Hq;
      // packed qkv offsets (uint4 units) of the two halves
      const int64_t pk = int64_t(t) * W + int64_t(head) * (D / 8) + g;
      // separate q / k tensors
      const int64_t sep = is_q ? (int64_t(t) * Hq + head) * (D / 8) + g
                               : (int64_t(t) * Hkv + (head - Hq)) * (D / 8) + g;
      float a[8], b[8], oa[8], ob[8];
      if (!BWD) {
        unpack8(src[pk], a);
        unpack8(src[pk + kG], b);
      } else {
        const uint4* s = is_q ? src : src_k;
        unpack8(s[sep], a);
        unpack8(s[sep + kG], b);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float c = cs[g * 8 + e], s = sn[g * 8 + e];
        oa[e] = a[e] * c - b[e] * s;
        ob[e] = b[e] * c + a[e] * s;
      }
      if (!BWD) {
        uint4* d = is_q ? dst : dst_k;
        d[sep] = pack8(oa);
        d[sep + kG] = pack8(ob);
      } else {
        dst[pk] = pack8(oa);
        dst[pk + kG] = pack8(ob);
      }
    }
    const int nv = Hkv * D / 8;
    for (int u = threadIdx.x; u < nv; u += blockDim.x) {
      const int64_t pk = int64_t(t) * W + int64_t(Hq + Hkv) * (D / 8) + u;
      const int64_t sep = int64_t(t) * nv + u;
      if (!BWD) dst_v[sep] = src[pk];
      else dst[pk] = src_v[sep];
    }
  }
}

__device__ __forceinline__ float sigmoid(float g) { return 1.f / (1.f + expf(-g)); }

// gu [rows, 2I] (gate columns, then up columns) -> m [rows, I] = silu(g) * u.
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const uint4* __restrict__ gu, uint4* __restrict__ m,
                                                         int64_t rows, int inter8) {
  const int64_t n = rows * inter8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / inter8;
    const int c = static_cast<int>(i - r * inter8);
    float g[8], u[8], o[8];
    unpack8(gu[r * 2 * inter8 + c], g);
    unpack8(gu[r * 2 * inter8 + inter8 + c], u);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = g[e] * sigmoid(g[e]) * u[e];
    m[i] = pack8(o);
  }
}

// dgu: dg = dm*u*s*(1 + g*(1-s)), du = dm*g*s with s = sigmoid(g).  dgu may
// alias gu (each element is read before it is written, by the same thread).
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const uint4* gu, const uint4* __restrict__ dm, uint4* dgu,
                                                         int64_t rows, int inter8) {
  const int64_t n = rows * inter8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / inter8;
    const int c = static_cast<int>(i - r * inter8);
    float g[8], u[8], d[8], og[8], ou[8];
    unpack8(gu[r * 2 * inter8 + c], g);
    unpack8(gu[r * 2 * inter8 + inter8 + c], u);
    unpack8(dm[i], d);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float s = sigmoid(g[e]);
      og[e] = d[e] * u[e] * s * (1.f + g[e] * (1.f - s));
      ou[e] = d[e] * g[e] * s;
    }
    dgu[r * 2 * inter8 + c] = pack8(og);
    dgu[r * 2 * inter8 + inter8 + c] = pack8(ou);
  }
}

int sm_count() {
  int dev = 0, n = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

int elementwise_grid(int64_t n) {
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = int64_t(sm_count()) * 8;
  return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

template <int NG>
cudaError_t norm_fwd_ng(const void* x, const void* w, void* y, float* rstd, int64_t rows, int groups, float eps,
                        cudaStream_t st) {
  const int64_t warps = rows;
  int64_t blocks = (warps + 3) / 4;
  const int64_t cap = int64_t(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  rmsnorm_fwd_kernel<NG><<<static_cast<int>(blocks), kNormThreads, 0, st>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(w), static_cast<uint4*>(y), rstd, rows, groups, eps);
  return cudaGetLastError();
}

template <int NG>
cudaError_t norm_dx_ng(const void* dy, const void* x, const void* w, const float* rstd, const void* dres, void* dx,
                       int64_t rows, int groups, cudaStream_t st) {
  int64_t blocks = (rows + 3) / 4;
  const int64_t cap = int64_t(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  rmsnorm_dx_kernel<NG><<<static_cast<int>(blocks), kNormThreads, 0, st>>>(
      static_cast<const uint4*>(dy), static_cast<const uint4*>(x), static_cast<const uint4*>(w), rstd,
      static_cast<const uint4*>(dres), static_cast<uint4*>(dx), rows, groups);
  return cudaGetLastError();
}

}  // namespace

int rmsnorm_bwd_blocks() { return sm_count() * 4; }

cudaError_t launch_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t rows, int hidden,
                               float eps, cudaStream_t st) {
  const int groups = hidden / 8;
  const int ng = (groups + 31) / 32;
  if (rows == 0) return cudaSuccess;
  if (ng <= 4) return norm_fwd_ng<4>(x, w, y, rstd, rows, groups, eps, st);
  if (ng <= 8) return norm_fwd_ng<8>(x, w, y, rstd, rows, groups, eps, st);
  if (ng <= 16) return norm_fwd_ng<16>(x, w, y, rstd, rows, groups, eps, st);
  if (ng <= 24) return norm_fwd_ng<24>(x, w, y, rstd, rows, groups, eps, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rmsnorm_bwd(const void* dy, const void* x, const void* w, const float* rstd, const void* dres,
                               void* dx, float* part, float* dw, int64_t rows, int hidden, cudaStream_t st) {
  const int groups = hidden / 8;
  const int ng = (groups + 31) / 32;
  const int nblocks = rmsnorm_bwd_blocks();
  cudaError_t e = cudaSuccess;
  if (rows > 0) {
    if (ng <= 4) e = norm_dx_ng<4>(dy, x, w, rstd, dres, dx, rows, groups, st);
    else if (ng <= 8) e = norm_dx_ng<8>(dy, x, w, rstd, dres, dx, rows, groups, st);
    else if (ng <= 16) e = norm_dx_ng<16>(dy, x, w, rstd, dres, dx, rows, groups, st);
    else if (ng <= 24) e = norm_dx_ng<24>(dy, x, w, rstd, dres, dx, rows, groups, st);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
  }
  rmsnorm_dw_kernel<<<nblocks, 256, 0, st>>>(static_cast<const uint4*>(dy), static_cast<const uint4*>(x), rstd, part,
                                             rows, groups);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  column_sum_kernel<<<(hidden + 255) / 256, 256, 0, st>>>(part, dw, nblocks, hidden);
  return cudaGetLastError();
}

cudaError_t launch_rope_split(const RowMap& map, const void* qkv, void* q, void* k, void* v, int T, int Hq, int Hkv,
                              int d, double rope_base, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int grid = T < sm_count() * 16 ? T : sm_count() * 16;
  const double lb = log2(rope_base);
  const uint4* s = static_cast<const uint4*>(qkv);
  if (d == 128)
    rope_kernel<128, false><<<grid, 128, 0, st>>>(map, s, nullptr, nullptr, static_cast<uint4*>(q),
                                                   static_cast<uint4*>(k), static_cast<uint4*>(v), T, Hq, Hkv, lb);
  else
    rope_kernel<64, false><<<grid, 128, 0, st>>>(map, s, nullptr, nullptr, static_cast<uint4*>(q),
                                                  static_cast<uint4*>(k), static_cast<uint4*>(v), T, Hq, Hkv, lb);
  return cudaGetLastError();
}

cudaError_t launch_rope_merge(const RowMap& map, const void* dq, const void* dk, const void* dv, void* dqkv, int T,
                              int Hq, int Hkv, int d, double rope_base, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int grid = T < sm_count() * 16 ? T : sm_count() * 16;
  const double lb = log2(rope_base);
  if (d == 128)
    rope_kernel<128, true><<<grid, 128, 0, st>>>(map, static_cast<const uint4*>(dq), static_cast<const uint4*>(dk),
                                                  static_cast<const uint4*>(dv), static_cast<uint4*>(dqkv), nullptr,
                                                  nullptr, T, Hq, Hkv, lb);
  else
    rope_kernel<64, true><<<grid, 128, 0, st>>>(map, static_cast<const uint4*>(dq), static_cast<const uint4*>(dk),
                                                 static_cast<const uint4*>(dv), static_cast<uint4*>(dqkv), nullptr,
                                                 nullptr, T, Hq, Hkv, lb);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_fwd(const void* gu, void* m, int64_t rows, int inter, cudaStream_t st) {
  const int64_t n = rows * (inter / 8);
  if (n == 0) return cudaSuccess;
  swiglu_fwd_kernel<<<elementwise_grid(n), 256, 0, st>>>(static_cast<const uint4*>(gu), static_cast<uint4*>(m), rows,
                                                         inter / 8);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const void* gu, const void* dm, void* dgu, int64_t rows, int inter, cudaStream_t st) {
  const int64_t n = rows * (inter / 8);
  if (n == 0) return cudaSuccess;
  swiglu_bwd_kernel<<<elementwise_grid(n), 256, 0, st>>>(static_cast<const uint4*>(gu), static_cast<const uint4*>(dm),
                                                         static_cast<uint4*>(dgu), rows, inter / 8);
  return cudaGetLastError();
}

}  // namespace dkv
