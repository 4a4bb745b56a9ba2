// Bandwidth-bound helpers of the backward pass: the D = rowsum(dO * O)
// preprocess (FlashAttention-2 backward, the lineage named on the DualKV
// research-map page) and the prompt dK/dV reduction + bf16 cast.
#include <cuda_bf16.h>

#include "checks.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {
namespace {

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(pa[i]);
    const float2 fb = __bfloat1622float2(pb[i]);
    s = fmaf(fa.x, fb.x, s);
    s = fmaf(fa.y, fb.y, s);
  }
  return s;
}

// LPR lanes cooperate on one row of d = 8*LPR features.
template <int LPR>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                         float* __restrict__ Dvec, int64_t rows, int T, int Hq,
                                                         float4* __restrict__ zero_ptr, int64_t zero_n4) {
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
  const int sub = threadIdx.x % LPR;
  // Every lane of a warp stays in the loop while any lane has a row, so the
  // shuffles below are always warp-convergent.
  for (int64_t r = tid / LPR; __any_sync(0xffffffffu, r < rows); r += nthreads / LPR) {
    float s = 0.f;
    if (r < rows) s = dot8_bf16(__ldg(o + r * LPR + sub), __ldg(dout + r * LPR + sub));
#pragma unroll
    for (int m = LPR / 2; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    if (sub == 0 && r < rows) {
      const int64_t t = r / Hq;
      const int h = static_cast<int>(r % Hq);
      Dvec[int64_t(h) * T + t] = s;
    }
  }
  for (int64_t i = tid; i < zero_n4; i += nthreads) zero_ptr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) prompt_reduce_kernel(const __grid_constant__ PromptMap map,
                                                            const float4* __restrict__ src_k,
                                                            const float4* __restrict__ src_v, int nsplit,
                                                            int64_t slice4, uint2* __restrict__ dk,
                                                            uint2* __restrict__ dv, float4* __restrict__ f32_k,
                                                            float4* __restrict__ f32_v, int row4,
                                                            unsigned int* err) {
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
  const int64_t n4 = int64_t(map.acc_row[map.ngroups]) * row4;
  for (int64_t i = tid; i < n4; i += nthreads) {
    const int32_t r = static_cast<int32_t>(i / row4);
    // group of accumulator row r: last g with acc_row[g] <= r
    int lo = 0, hi = map.ngroups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (map.acc_row[mid] <= r) lo = mid; else hi = mid - 1;
    }
    if (!check(r >= map.acc_row[lo] && r < map.acc_row[lo + 1], err, 1301)) continue;
    const int64_t out = (int64_t(map.packed_row[lo]) + (r - map.acc_row[lo])) * row4 + (i - int64_t(r) * row4);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float4* src = which ? src_v : src_k;
      float4 a = src[i];
      for (int sp = 1; sp < nsplit; ++sp) {
        const float4 b = src[sp * slice4 + i];
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(a.x, a.y);
      __nv_bfloat162 hi2 = __floats2bfloat162_rn(a.z, a.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo2);
      pk.y = *reinterpret_cast<uint32_t*>(&hi2);
      (which ? dv : dk)[out] = pk;
      float4* f32 = which ? f32_v : f32_k;
      if (f32 != nullptr) f32[i] = a;
    }
  }
}

// dq = scale * dq_acc, transposed from [Hq][D/4][T][4] to [T][Hq][D]: one
// block per 32 rows of one head, staged through shared memory so that both
// the reads (32 consecutive rows of a 4-column chunk) and the writes (whole
// rows of the head) are contiguous.
template <int D>
__global__ void __launch_bounds__(256) dq_cast_kernel(const float4* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                      float* __restrict__ dq_prompt, int64_t T, int Hq, float scale,
                                                      int64_t prompt_end, int64_t keep_lo, int64_t keep_hi) {
  __shared__ float4 tile[32][D / 4 + 1];
  const int h = blockIdx.y;
  const int64_t t0 = int64_t(blockIdx.x) * 32;
  const int tid = threadIdx.x;
  for (int c = tid / 32; c < D / 4; c += 8) {
    const int64_t t = t0 + (tid % 32);
    tile[tid % 32][c] = t < T ? acc[(int64_t(h) * (D / 4) + c) * T + t] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  constexpr int kParts = D / 16;  // 16 columns per thread
  for (int i = tid; i < 32 * kParts; i += 256) {
    const int r = i / kParts, part = i % kParts;
    const int64_t t = t0 + r;
    if (t >= T || (t < prompt_end && (t < keep_lo || t >= keep_hi))) continue;
    float f[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 v = tile[r][part * 4 + u];
      f[4 * u] = v.x * scale;
      f[4 * u + 1] = v.y * scale;
      f[4 * u + 2] = v.z * scale;
      f[4 * u + 3] = v.w * scale;
    }
    uint4* dst = reinterpret_cast<uint4*>(dq + (t * Hq + h) * D + part * 16);
    dst[0] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                        pack_bf16x2(f[6], f[7]));
    dst[1] = make_uint4(pack_bf16x2(f[8], f[9]), pack_bf16x2(f[10], f[11]), pack_bf16x2(f[12], f[13]),
                        pack_bf16x2(f[14], f[15]));
    if (dq_prompt != nullptr && t < prompt_end) {
      float4* d32 = reinterpret_cast<float4*>(dq_prompt + (t * Hq + h) * D + part * 16);
#pragma unroll
      for (int u = 0; u < 4; ++u) d32[u] = make_float4(f[4 * u], f[4 * u + 1], f[4 * u + 2], f[4 * u + 3]);
    }
  }
}

// One thread waits, with the kernels' own bounded wait, for an mbarrier
// phase that nothing completes; the wait gives up after limit_ns, records a
// timeout at `site` in the error word and the kernel returns normally.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(unsigned int* err, uint64_t limit_ns,
                                                                  uint32_t site) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, err, site, limit_ns);
  }
}

int grid_for(int64_t work_threads) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (work_threads + 255) / 256;
  const int64_t cap = int64_t(sms) * 8;  // 8 resident 256-thread blocks per SM
  return static_cast<int>(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace

cudaError_t launch_preprocess(const void* out, const void* dout, float* Dvec, int64_t T, int Hq, int d,
                              float* zero_ptr, size_t zero_n, cudaStream_t stream) {
  const int64_t rows = T * Hq;
  const int lpr = d / 8;
  const int grid = grid_for(rows * lpr);
  const int64_t z4 = static_cast<int64_t>(zero_n / 4);
  if (lpr == 16)
    preprocess_kernel<16><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(out), static_cast<const uint4*>(dout),
                                                    Dvec, rows, static_cast<int>(T), Hq,
                                                    reinterpret_cast<float4*>(zero_ptr), z4);
  else
    preprocess_kernel<8><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(out), static_cast<const uint4*>(dout),
                                                   Dvec, rows, static_cast<int>(T), Hq,
                                                   reinterpret_cast<float4*>(zero_ptr), z4);
  return cudaGetLastError();
}

cudaError_t launch_dq_cast(const float* dq_acc, void* dq, float* dq_prompt, int64_t T, int Hq, int d, float scale,
                           int64_t prompt_end, int64_t keep_lo, int64_t keep_hi, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((T + 31) / 32), static_cast<unsigned>(Hq));
  if (d == 64)
    dq_cast_kernel<64><<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc),
                                                 static_cast<__nv_bfloat16*>(dq), dq_prompt, T, Hq, scale, prompt_end,
                                                 keep_lo, keep_hi);
  else
    dq_cast_kernel<128><<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc),
                                                  static_cast<__nv_bfloat16*>(dq), dq_prompt, T, Hq, scale,
                                                  prompt_end, keep_lo, keep_hi);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned int* err, uint64_t limit_ns, uint32_t site, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns, site);
  return cudaGetLastError();
}

cudaError_t launch_prompt_reduce(const float* src_k, const float* src_v, int nsplit, size_t slice, void* dk,
                                 void* dv, float* f32_k, float* f32_v, const PromptMap& map, int row_elems,
                                 unsigned int* err, cudaStream_t stream) {
  if (map.ngroups == 0) return cudaSuccess;
  const int row4 = row_elems / 4;
  const int64_t n4 = int64_t(map.acc_row[map.ngroups]) * row4;
  if (n4 == 0) return cudaSuccess;
  prompt_reduce_kernel<<<grid_for(n4), 256, 0, stream>>>(
      map, reinterpret_cast<const float4*>(src_k), reinterpret_cast<const float4*>(src_v), nsplit,
      static_cast<int64_t>(slice / 4), static_cast<uint2*>(dk), static_cast<uint2*>(dv),
      reinterpret_cast<float4*>(f32_k), reinterpret_cast<float4*>(f32_v), row4, err);
  return cudaGetLastError();
}

}  // namespace dkv
