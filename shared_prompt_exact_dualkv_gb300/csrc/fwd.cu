// Forward kernel: exact attention over the packed shared-prompt layout.
//
// One CTA computes one 128-row query tile of one q-head.  Its key loop walks
// two disjoint regions in the same launch (DualKV research-map page,
// "Approach"; forum page, "Two changes", change 1): the shared prompt keys,
// then the causal keys of the query's own response.  QK^T and PV run on the
// tcgen05 tensor cores with TMEM accumulators; the softmax is online
// (running max and sum, FlashAttention-2 lineage named on the research-map
// page) and the kernel writes O (bf16) and the natural-log LSE (fp32).
//
// Warp roles (320 threads):
//   warps 0-7  softmax + epilogue; warp w owns query rows 32*(w%4) .. +31 (its
//              TMEM lane quarter) and key columns 64*(w/4) .. +63 of each S
//              tile, so every row is shared by two threads that swap their
//              partial row maxima through shared memory once per key tile
//   warp  8    TMA producer: Q once, then K/V tiles into 2-stage rings
//   warp  9    TMEM allocator and MMA issuer
// TMEM columns: S double buffer [0,128) and [128,256), O [256,256+D),
// P (bf16, two per column) [384,448).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kX = kV + kStages * kTileBytes;  // row-max exchange [2][2][128] + row sums [2][128]
  static constexpr int kBar = kX + 3072;
  static constexpr int kBytes = kBar + 256 + 1024;  // barriers, TMEM slot, alignment slack
};

enum FwdBar {
  kQFull = 0,
  kKFull = 1,     // + stage
  kVFull = 3,     // + stage
  kKEmpty = 5,    // + stage: released once QK^T has read it
  kVEmpty = 7,    // + stage: released once PV has read it
  kSFull = 9,     // + buffer
  kSFree = 11,    // + buffer
  kPFull = 13,
  kODone = 14,
  kXch = 15,      // + tile parity: both halves of every row posted their max
  kLx = 17,       // both halves posted their row sums
  kNumFwdBars = 18
};

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP = 384;
constexpr int kSmThreads = 256;  // softmax threads (two per query row)

template <int D>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ Sched s, const __grid_constant__ CUtensorMap mQ,
               const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
               __nv_bfloat16* __restrict__ out, float* __restrict__ lse, unsigned int* err) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kBar + 192);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t item = s.items[blockIdx.x / s.Hq];
  const int h = blockIdx.x % s.Hq;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kKFull + i], 1);
      mbar_init(&bar[kVFull + i], 1);
      mbar_init(&bar[kKEmpty + i], 1);
      mbar_init(&bar[kVEmpty + i], 1);
      mbar_init(&bar[kSFull + i], 1);
      mbar_init(&bar[kSFree + i], kSmThreads);
      mbar_init(&bar[kXch + i], kSmThreads);
    }
    mbar_init(&bar[kPFull], kSmThreads);
    mbar_init(&bar[kODone], 1);
    mbar_init(&bar[kLx], kSmThreads);
    fence_mbar_init();
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    // The warp runs the loop converged; one elected lane issues each copy.
    {
      if (elect_one()) {
        mbar_arrive_expect_tx(&bar[kQFull], L::kTileBytes);
        for (int a = 0; a < D / 64; ++a) tma_load_3d(sm + L::kQ + a * 16384, &mQ, &bar[kQFull], a * 64, h, w.q0);
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        const int k0 = w.k0(j);
        uint8_t* sK = sm + L::kK + st * L::kTileBytes;
        uint8_t* sV = sm + L::kV + st * L::kTileBytes;
        if (j >= 2 && !mbar_wait(&bar[kKEmpty + st], ((j >> 1) - 1) & 1, err, 101)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kKFull + st], L::kTileBytes);
          for (int a = 0; a < D / 64; ++a) tma_load_3d(sK + a * 16384, &mK, &bar[kKFull + st], a * 64, hk, k0);
        }
        k_issued = j + 1;
        if (j >= 2 && !mbar_wait(&bar[kVEmpty + st], ((j >> 1) - 1) & 1, err, 102)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kVFull + st], L::kTileBytes);
          for (int a = 0; a < D / 64; ++a) tma_load_3d(sV + a * 16384, &mV, &bar[kVFull + st], a * 64, hk, k0);
        }
        v_issued = j + 1;
      }
      // Before the CTA can exit, every copy this warp issued must have landed
      // (the consumers may have stopped early on an error).
      for (int j = (k_issued > 2 ? k_issued - 2 : 0); j < k_issued; ++j)
        mbar_wait(&bar[kKFull + (j & 1)], (j >> 1) & 1, err, 103);
      for (int j = (v_issued > 2 ? v_issued - 2 : 0); j < v_issued; ++j)
        mbar_wait(&bar[kVFull + (j & 1)], (j >> 1) & 1, err, 104);
      mbar_wait(&bar[kQFull], 0, err, 105);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // The warp runs the loop converged (warp-uniform control flow and
    // descriptors); one elected lane issues each MMA and commit.
    {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(sm + L::kQ);
      bool ok = mbar_wait(&bar[kQFull], 0, err, 201);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&bar[kKFull + st], (j >> 1) & 1, err, 202)) return false;
        if (j >= 2 && !mbar_wait(&bar[kSFree + st], ((j >> 1) - 1) & 1, err, 203)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + L::kK + st * L::kTileBytes);
        const uint32_t dS = tmem + (st ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (elect_one()) mma_ss(dS, desc_kmajor_sw128(sQ + off), desc_kmajor_sw128(sK + off), idS, kk > 0 ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kSFull + st]);
        if (elect_one()) mma_commit(&bar[kKEmpty + st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j & 1;
        if (j + 1 < n && !issue_s(j + 1)) break;
        if (!mbar_wait(&bar[kPFull], j & 1, err, 204)) break;
        if (!mbar_wait(&bar[kVFull + st], (j >> 1) & 1, err, 205)) break;
        tc_fence_after();
        const uint32_t sV = smem_u32(sm + L::kV + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (elect_one()) mma_ts(tmem + kColO, tmem + kColP + kk * 8, desc_mnmajor_sw128(sV + kk * 2048, 16384), idO,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kODone]);
        if (elect_one()) mma_commit(&bar[kVEmpty + st]);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int cb = half * 64;  // first key column of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float* xmax = reinterpret_cast<float*>(sm + L::kX);  // [parity][half][row]
    float* xsum = xmax + 512;                            // [half][row]
    const float c = s.scale_log2;
    float m_use = -INFINITY;
    float l = 0.f;  // this thread's share of the row sum
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&bar[kSFull + b], (j >> 1) & 1, err, 301)) { ok = false; break; }
      tc_fence_after();
      float x[64];
      {
        const uint32_t tS = tmem + lane_off + (b ? kColS1 : kColS0) + cb;
        uint32_t r[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(&bar[kSFree + b]);

      const int mk = w.mask_kind(j);
      if (mk == 1) {
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (cb + i > row) ? -INFINITY : x[i];
      } else if (mk == 2) {
        const int lim = w.P - w.k0(j) - cb;
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (i >= lim) ? -INFINITY : x[i];
      }
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
      for (int i = 8; i < 64; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // row maximum over both halves of the tile
      xmax[(b * 2 + half) * 128 + row] = mt;
      mbar_arrive(&bar[kXch + b]);
      if (!mbar_wait(&bar[kXch + b], (j >> 1) & 1, err, 304)) { ok = false; break; }
      mt = fmaxf(mt, xmax[(b * 2 + (half ^ 1)) * 128 + row]);
      const float m_cand = mt * c;
      // Keep the running maximum unless it grows by more than 2^8: the final
      // normalisation is exact for any reference value, and skipping the
      // rescale keeps O in TMEM untouched on most tiles.
      const bool resc = m_cand > m_use + 8.f;
      const float m_new = resc ? m_cand : m_use;
      const float alpha = resc ? ex2(m_use - m_new) : 1.f;
      const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
      uint32_t p[32];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float e0 = ex2(fmaf(x[2 * i], c, -m_sub));
        const float e1 = ex2(fmaf(x[2 * i + 1], c, -m_sub));
        rs[i & 3] += e0 + e1;
        p[i] = pack_bf16x2(e0, e1);
      }
      // The previous PV product must be done before P is overwritten and O rescaled.
      if (j > 0) {
        if (!mbar_wait(&bar[kODone], (j - 1) & 1, err, 302)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
          const uint32_t tO = tmem + lane_off + kColO + half * (D / 2);
#pragma unroll
          for (int ci = 0; ci < D / 64; ++ci) {
            uint32_t r[32];
            tmem_ld32(tO + ci * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + ci * 32, r);
          }
        }
      }
      l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      m_use = m_new;
      tmem_st32(tmem + lane_off + kColP + half * 32, p);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[kPFull]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&bar[kODone], (n - 1) & 1, err, 303);
    if (ok) {
      xsum[half * 128 + row] = l;
      mbar_arrive(&bar[kLx]);
      ok = mbar_wait(&bar[kLx], 0, err, 305);
      if (ok) l += xsum[(half ^ 1) * 128 + row];
    }
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int q = w.q0 + row;
      const bool valid = q < w.q_end;
      const float inv_l = 1.f / l;
      const uint32_t tO = tmem + lane_off + kColO + half * (D / 2);
      uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(q) * s.Hq + h) * D + half * (D / 2));
#pragma unroll
      for (int ci = 0; ci < D / 64; ++ci) {
        uint32_t r[32];
        tmem_ld32(tO + ci * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[ci * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (valid && half == 0) lse[static_cast<size_t>(h) * s.T + q] = (m_use + log2f(l)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
static cudaError_t launch_fwd_d(const Sched& s, const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, void* out, float* lse, unsigned int* err,
                                cudaStream_t stream) {
  using L = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(s.num_items) * static_cast<unsigned>(s.Hq);
  fwd_kernel<D><<<grid, 320, L::kBytes, stream>>>(s, mQ, mK, mV, static_cast<__nv_bfloat16*>(out), lse, err);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK,
                       const CUtensorMap& mV, void* out, float* lse, unsigned int* err, cudaStream_t stream) {
  if (s.num_items == 0) return cudaSuccess;
  return d == 64 ? launch_fwd_d<64>(s, mQ, mK, mV, out, lse, err, stream)
                 : launch_fwd_d<128>(s, mQ, mK, mV, out, lse, err, stream);
}

}  // namespace dkv
