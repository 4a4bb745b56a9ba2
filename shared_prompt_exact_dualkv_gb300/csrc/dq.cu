// dQ kernel of the backward pass.
//
// One CTA owns one 128-row query tile of one q-head and walks the same two
// key regions as the forward (shared prompt, then the query's own response;
// DualKV research-map page, "Approach").  Per key tile it recomputes the
// probabilities from the saved LSE (FlashAttention-2 style backward, the
// lineage named on the research-map page):
//   S = Q K^T, P = exp(scale*S - LSE), dP = dO V^T, dS = P * (dP - D),
//   dQ += dS K,   and finally dQ *= scale.
// A CTA is the only writer of its dQ rows, so dQ needs no atomics.
//
// Warp roles (320 threads): warps 0-7 elementwise -- warp w handles query
// rows 32*(w%4) .. +31 (its TMEM lane quarter) and key columns 64*(w/4) .. +63,
// so every SM sub-partition runs two elementwise warps; warp 8 TMA producer;
// warp 9 TMEM allocator + MMA issuer.
// TMEM columns: S [0,128), dP [128,256), dQ [256,256+D), dS (bf16, two per
// column) double buffer [384,448) and [448,512).
#include <cuda_bf16.h>

#include "checks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {
namespace {

template <int D>
struct DqLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kTileBytes;
  static constexpr int kK = kdO + kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kBar = kV + kVStages * kTileBytes;
  static constexpr int kBytes = kBar + 256 + 1024;
};

enum DqBar {
  kQFull = 0,
  kKFull = 1,    // + stage (3)
  kKEmpty = 4,   // + stage (3)
  kVFull = 7,    // + stage (2)
  kVEmpty = 9,   // + stage (2)
  kSFull = 11,
  kSFree = 12,
  kdPFull = 13,
  kdPFree = 14,
  kdSFull = 15,  // + buffer (2)
  kdSFree = 17,  // + buffer (2)
  kNumDqBars = 19
};

constexpr uint32_t kColS = 0, kColdP = 128, kColdQ = 256, kColdS = 384;
constexpr int kEwThreads = 256;

template <int D>
__global__ void __launch_bounds__(320, 1)
    dq_kernel(const __grid_constant__ Sched s, const __grid_constant__ CUtensorMap mQ,
              const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
              const __grid_constant__ CUtensorMap mdO, const float* __restrict__ lse,
              const float* __restrict__ Dvec, __nv_bfloat16* __restrict__ dq, float* __restrict__ dq_prompt,
              unsigned int* err) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kBar + 192);
  const RoleSteps steps{reinterpret_cast<int32_t*>(sm + L::kBar + 200)};  // checks build only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t item = s.items[s.heads_outer ? blockIdx.x % s.num_items : blockIdx.x / s.Hq];
  const int h = s.heads_outer ? blockIdx.x / s.num_items : blockIdx.x % s.Hq;
  const int hk = h / s.group;
  KeyWalk w;
  w.init(s, item);
  const int n = w.n;

  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    mbar_init(&bar[kQFull], 1);
    for (int i = 0; i < L::kKStages; ++i) {
      mbar_init(&bar[kKFull + i], 1);
      mbar_init(&bar[kKEmpty + i], 1);
    }
    for (int i = 0; i < L::kVStages; ++i) {
      mbar_init(&bar[kVFull + i], 1);
      mbar_init(&bar[kVEmpty + i], 1);
    }
    mbar_init(&bar[kSFull], 1);
    mbar_init(&bar[kSFree], kEwThreads);
    mbar_init(&bar[kdPFull], 1);
    mbar_init(&bar[kdPFree], kEwThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kdSFull + i], kEwThreads);
      mbar_init(&bar[kdSFree + i], 1);
    }
    fence_mbar_init();
    steps.init();
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    // The warp runs the loop converged; one elected lane issues each copy.
    {
      // (an out-of-range tile copy would only read zeros; the checks record it)
      check(w.q0 >= 0 && w.q0 < s.T && h < s.Hq, err, 1201);
      if (elect_one()) {
        mbar_arrive_expect_tx(&bar[kQFull], 2 * L::kTileBytes);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(sm + L::kQ + a * 16384, &mQ, &bar[kQFull], a * 64, h, w.q0);
          tma_load_3d(sm + L::kdO + a * 16384, &mdO, &bar[kQFull], a * 64, h, w.q0);
        }
      }
      int ks = 0, kph = 0, vs = 0, vph = 0, k_issued = 0, v_issued = 0;
      for (int j = 0; j < n; ++j) {
        const int k0 = w.k0(j);
        check(k0 >= 0 && k0 < s.T && hk < s.Hkv, err, 1202);
        if (j >= L::kKStages && !mbar_wait(&bar[kKEmpty + ks], kph ^ 1, err, 401)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kKFull + ks], L::kTileBytes);
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sm + L::kK + ks * L::kTileBytes + a * 16384, &mK, &bar[kKFull + ks], a * 64, hk, k0);
        }
        k_issued = j + 1;
        if (j >= L::kVStages && !mbar_wait(&bar[kVEmpty + vs], vph ^ 1, err, 402)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kVFull + vs], L::kTileBytes);
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sm + L::kV + vs * L::kTileBytes + a * 16384, &mV, &bar[kVFull + vs], a * 64, hk, k0);
        }
        v_issued = j + 1;
        if (++ks == L::kKStages) { ks = 0; kph ^= 1; }
        if (++vs == L::kVStages) { vs = 0; vph ^= 1; }
      }
      if (lane == 0) steps.put(0, v_issued);
      // Before the CTA can exit, every copy this warp issued must have landed
      // (the consumers may have stopped early on an error).
      for (int j = (k_issued > L::kKStages ? k_issued - L::kKStages : 0); j < k_issued; ++j)
        mbar_wait(&bar[kKFull + j % L::kKStages], (j / L::kKStages) & 1, err, 403);
      for (int j = (v_issued > L::kVStages ? v_issued - L::kVStages : 0); j < v_issued; ++j)
        mbar_wait(&bar[kVFull + j % L::kVStages], (j / L::kVStages) & 1, err, 404);
      mbar_wait(&bar[kQFull], 0, err, 405);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // The warp runs the loop converged (warp-uniform control flow and
    // descriptors); one elected lane issues each MMA and commit.
    {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idQ = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(sm + L::kQ);
      const uint32_t sdO = smem_u32(sm + L::kdO);
      bool ok = mbar_wait(&bar[kQFull], 0, err, 501);
      // S_j = Q K_j^T and dP_j = dO V_j^T
      auto issue_s = [&](int j) -> bool {
        const int ks = j % L::kKStages;
        if (!mbar_wait(&bar[kKFull + ks], (j / L::kKStages) & 1, err, 502)) return false;
        if (j >= 1 && !mbar_wait(&bar[kSFree], (j - 1) & 1, err, 503)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (elect_one()) mma_ss(tmem + kColS, desc_kmajor_sw128(sQ + off), desc_kmajor_sw128(sK + off), idSS, kk > 0 ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kSFull]);
        return true;
      };
      auto issue_dp = [&](int j) -> bool {
        const int vs = j % L::kVStages;
        if (!mbar_wait(&bar[kVFull + vs], (j / L::kVStages) & 1, err, 504)) return false;
        if (j >= 1 && !mbar_wait(&bar[kdPFree], (j - 1) & 1, err, 505)) return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(sm + L::kV + vs * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (elect_one()) mma_ss(tmem + kColdP, desc_kmajor_sw128(sdO + off), desc_kmajor_sw128(sV + off), idSS, kk > 0 ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kdPFull]);
        if (elect_one()) mma_commit(&bar[kVEmpty + vs]);
        return true;
      };
      if (ok) ok = issue_s(0) && issue_dp(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !(issue_s(j + 1) && issue_dp(j + 1))) break;
        const int b = j & 1;
        if (!mbar_wait(&bar[kdSFull + b], (j >> 1) & 1, err, 506)) break;
        tc_fence_after();
        const int ks = j % L::kKStages;
        const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (elect_one()) mma_ts(tmem + kColdQ, tmem + kColdS + b * 64 + kk * 8, desc_mnmajor_sw128(sK + kk * 2048, 16384), idQ,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kdSFree + b]);
        if (elect_one()) mma_commit(&bar[kKEmpty + ks]);
        if (lane == 0) steps.put(1, j + 1);
      }
    }
  } else {
    // ---------------------------------------------------------------- elementwise
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int cb = half * 64;  // first key column of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    const int q = w.q0 + row;
    // Rows past the segment end are never stored; give them P = 0.
    float lse2 = INFINITY, Dr = 0.f;
    if (q < w.q_end && check_index(static_cast<int64_t>(h) * s.T + q, static_cast<int64_t>(s.Hq) * s.T, err, 1203)) {
      lse2 = lse[static_cast<size_t>(h) * s.T + q] * 1.4426950408889634f;
      Dr = Dvec[static_cast<size_t>(h) * s.T + q];
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&bar[kSFull], j & 1, err, 601)) { ok = false; break; }
      tc_fence_after();
      float p[64];
      {
        uint32_t r[64];
        tmem_ld32(tmem + lane_off + kColS + cb, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(tmem + lane_off + kColS + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) p[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(&bar[kSFree]);
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 a = fma2(make_float2(p[i], p[i + 1]), make_float2(c, c), make_float2(-lse2, -lse2));
        p[i] = ex2(a.x);
        p[i + 1] = ex2(a.y);
      }
      const int mk = w.mask_kind(j);
      if (mk == 1) {
#pragma unroll
        for (int i = 0; i < 64; ++i) p[i] = (cb + i > row) ? 0.f : p[i];
      } else if (mk == 2) {
        const int lim = w.key_limit(j) - cb;
#pragma unroll
        for (int i = 0; i < 64; ++i) p[i] = (i >= lim) ? 0.f : p[i];
      }
      if (!mbar_wait(&bar[kdPFull], j & 1, err, 602)) { ok = false; break; }
      tc_fence_after();
      // dS buffer b was last read by the dQ product of tile j-2.
      if (j >= 2 && !mbar_wait(&bar[kdSFree + b], ((j >> 1) - 1) & 1, err, 603)) { ok = false; break; }
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kColdP + cb + ci * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 t = add2(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                make_float2(-Dr, -Dr));
          const float2 ds = mul2(make_float2(p[ci * 32 + 2 * i], p[ci * 32 + 2 * i + 1]), t);
          pk[i] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st16(tmem + lane_off + kColdS + b * 64 + half * 32 + ci * 16, pk);
      }
      tc_fence_before();
      mbar_arrive(&bar[kdPFree]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[kdSFull + b]);
      if (row == 0) steps.put(2 + half, j + 1);
    }
    // ---------------------------------------------------------------- epilogue
    const int bl = (n - 1) & 1;
    if (ok) ok = n > 0 && mbar_wait(&bar[kdSFree + bl], ((n - 1) >> 1) & 1, err, 604);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const bool valid = q < w.q_end;
      uint4* dst = reinterpret_cast<uint4*>(dq + (static_cast<size_t>(q) * s.Hq + h) * D + half * (D / 2));
      // A prompt row's fp32 dQ also goes to dq_prompt (accumulator row order,
      // [prompt rows of all groups, Hq, D]) when the caller asked for it.
      const int32_t seg = static_cast<int32_t>(item_seg(item));
      float4* dst32 = nullptr;
      if (dq_prompt != nullptr && s.prompt_of(seg) == seg &&
          (!valid || check(s.acc_row[seg] + (q - s.off[seg]) < s.acc_rows, err, 1205)))
        dst32 = reinterpret_cast<float4*>(
            dq_prompt + (static_cast<size_t>(s.acc_row[seg] + (q - s.off[seg])) * s.Hq + h) * D + half * (D / 2));
#pragma unroll
      for (int ci = 0; ci < D / 64; ++ci) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kColdQ + half * (D / 2) + ci * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * s.scale, __uint_as_float(r[2 * i + 1]) * s.scale);
        if (valid && check(q >= 0 && q < s.T && h < s.Hq, err, 1204)) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[ci * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          if (dst32 != nullptr) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst32[ci * 8 + v] = make_float4(__uint_as_float(r[4 * v]) * s.scale, __uint_as_float(r[4 * v + 1]) * s.scale,
                                              __uint_as_float(r[4 * v + 2]) * s.scale, __uint_as_float(r[4 * v + 3]) * s.scale);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 256) steps.verify(n, err, 1206);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_dq_d(const Sched& s, const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                        const CUtensorMap& mdO, const float* lse, const float* Dvec, void* dq, float* dq_prompt,
                        unsigned int* err, cudaStream_t stream) {
  using L = DqLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(s.num_items) * static_cast<unsigned>(s.Hq);
  dq_kernel<D><<<grid, 320, L::kBytes, stream>>>(s, mQ, mK, mV, mdO, lse, Dvec, static_cast<__nv_bfloat16*>(dq),
                                                 dq_prompt, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                      const CUtensorMap& mdO, const float* lse, const float* Dvec, void* dq, float* dq_prompt,
                      unsigned int* err, cudaStream_t stream) {
  if (s.num_items == 0) return cudaSuccess;
  return d == 64 ? launch_dq_d<64>(s, mQ, mK, mV, mdO, lse, Dvec, dq, dq_prompt, err, stream)
                 : launch_dq_d<128>(s, mQ, mK, mV, mdO, lse, Dvec, dq, dq_prompt, err, stream);
}

}  // namespace dkv
