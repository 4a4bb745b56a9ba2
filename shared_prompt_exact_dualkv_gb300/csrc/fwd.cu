// Forward kernel: exact attention over the packed shared-prompt layout.
//
// One CTA computes one 128-row query tile for two q-heads of the same GQA
// group (or one head when the group size is odd).  Its key loop walks two
// disjoint regions in the same launch (DualKV research-map page, "Approach";
// forum page, "Two changes", change 1): the shared prompt keys, then the
// causal keys of the query's own response.  QK^T and PV run on the tcgen05
// tensor cores with TMEM accumulators; the softmax is online (running max and
// sum, FlashAttention-2 lineage named on the research-map page) and the
// kernel writes O (bf16) and the natural-log LSE (fp32).
//
// The two heads share every K/V tile (one copy from L2 feeds both) and form a
// ping-pong: while the softmax of head A works on its scores, the tensor
// cores run head B's products and vice versa.  Per key tile j the MMA stream
// is PV_A(j) S_A(j+1) PV_B(j) S_B(j+1).
// Warp roles (320 threads):
//   warps 0-3  softmax + epilogue of head A (thread r owns query row r)
//   warps 4-7  softmax + epilogue of head B
//   warp  8    TMA producer: both Q tiles once, then K and V tiles into 2-stage rings
//   warp  9    TMEM allocator and MMA issuer
// Producer and MMA warps run their loops converged; one elected lane issues
// each copy, MMA and commit.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [384,384+D).
// P (bf16, two per column) overwrites the first 64 columns of its head's S
// block once the softmax has read it; the next S of that head is issued after
// the PV product that reads P.
#include <cuda_bf16.h>

#include "checks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kKS = 2;  // K ring depth
  static constexpr int kVS = 2;  // V ring depth
  static constexpr int kQ = 0;   // two Q tiles (heads A, B)
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kKS * kTileBytes;
  static constexpr int kBar = kV + kVS * kTileBytes;
  static constexpr int kBytes = kBar + 256 + 1024;  // barriers, TMEM slot, alignment slack
};

enum FwdBar {
  kQFull = 0,
  kKFull = 1,     // + stage (3)
  kKEmpty = 4,    // + stage: released once both heads' QK^T have read it
  kVFull = 7,     // + stage (2)
  kVEmpty = 9,    // + stage: released once both heads' PV have read it
  kSFull = 11,    // + head: scores of the current key tile are in TMEM
  kPFull = 13,    // + head: P written to TMEM (and O rescaled)
  kODone = 15,    // + head: last PV product complete
  kNumFwdBars = 17
};

constexpr int kHeadThreads = 128;

__device__ __forceinline__ uint32_t col_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }

// Heads of one CTA: (2*slot, 2*slot+1) when the group size is even, else one.
__host__ __device__ inline int fwd_head_slots(int Hq, int group) { return (group % 2 == 0) ? Hq / 2 : Hq; }

// Row maximum of 128 scores read from TMEM in two 64-column halves; columns
// >= lim are excluded (lim = 128 on unmasked tiles).
template <bool MASKED>
__device__ __forceinline__ float row_max(uint32_t tS, int lim) {
  if constexpr (!MASKED) {
    // the TMEM load reduces each thread's 32 columns itself
    float m = -INFINITY;
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      uint32_t r[64];
      const float m0 = tmem_ld32_max(tS + hc * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
      const float m1 = tmem_ld32_max(tS + hc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
      tmem_ld_wait();
      m = fmax3(m, m0, m1);
    }
    return m;
  } else {
    float mx[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      uint32_t r[64];
      tmem_ld32(tS + hc * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
      tmem_ld32(tS + hc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float v0 = (hc * 64 + i < lim) ? __uint_as_float(r[i]) : -INFINITY;
        const float v1 = (hc * 64 + i + 1 < lim) ? __uint_as_float(r[i + 1]) : -INFINITY;
        mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], v0, v1);
      }
    }
    return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
  }
}

// P = exp2(c*S - m_sub) as bf16 written over the first 64 columns of S.
// Returns the row sums of the probabilities before (.x) and after (.y)
// rounding to bf16: PV multiplies the rounded values, so O is normalised by
// their sum (the weights then add up to one), while the LSE keeps the exact
// sum.
template <bool MASKED>
__device__ __forceinline__ float2 row_exp(uint32_t tS, int lim, float c, float m_sub) {
  float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float rr_lo = 0.f, rr_hi = 0.f;
  const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_sub, -m_sub);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    uint32_t r[64];
    tmem_ld32(tS + hc * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld32(tS + hc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld_wait();
    uint32_t p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int cc = hc * 64 + 2 * i;
      const float2 a = fma2(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, nm2);
      float2 e = make_float2(ex2(a.x), ex2(a.y));
      if (MASKED) {
        e.x = (cc < lim) ? e.x : 0.f;
        e.y = (cc + 1 < lim) ? e.y : 0.f;
      }
      rs[i & 3] = add2(rs[i & 3], e);
      p[i] = pack_bf16x2(e.x, e.y);
      add_bf16x2_f32(rr_lo, rr_hi, p[i]);
    }
    tmem_st32(tS + hc * 32, p);
  }
  const float2 t = add2(add2(rs[0], rs[1]), add2(rs[2], rs[3]));
  return make_float2(t.x + t.y, rr_lo + rr_hi);
}

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
  const RoleSteps steps{reinterpret_cast<int32_t*>(sm + L::kBar + 200)};  // checks build only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slots = fwd_head_slots(s.Hq, s.group);
  const uint32_t item = s.items[s.heads_outer ? blockIdx.x % s.num_items : blockIdx.x / slots];
  const int slot = s.heads_outer ? blockIdx.x / s.num_items : blockIdx.x % slots;
  const bool paired = (s.group % 2 == 0);
  const int nheads = paired ? 2 : 1;
  const int h0 = paired ? 2 * slot : slot;  // head A; head B = h0 + 1
  const int hk = h0 / s.group;
  KeyWalk w;
  w.init(s, item);
  const int n = w.n;

  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    mbar_init(&bar[kQFull], 1);
    for (int i = 0; i < L::kKS; ++i) {
      mbar_init(&bar[kKFull + i], 1);
      mbar_init(&bar[kKEmpty + i], 1);
    }
    for (int i = 0; i < L::kVS; ++i) {
      mbar_init(&bar[kVFull + i], 1);
      mbar_init(&bar[kVEmpty + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kSFull + i], 1);
      mbar_init(&bar[kPFull + i], kHeadThreads / 32);  // one arrival per softmax warp
      mbar_init(&bar[kODone + i], 1);
    }
    fence_mbar_init();
    steps.init();
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
    // (an out-of-range tile copy would only read zeros; the checks record it)
    check(w.q0 >= 0 && w.q0 < s.T && h0 + nheads <= s.Hq, err, 1001);
    if (elect_one()) {
      mbar_arrive_expect_tx(&bar[kQFull], nheads * L::kTileBytes);
      for (int x = 0; x < nheads; ++x)
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sm + L::kQ + x * L::kTileBytes + a * 16384, &mQ, &bar[kQFull], a * 64, h0 + x, w.q0);
    }
    int k_issued = 0, v_issued = 0;
    for (int j = 0; j < n; ++j) {
      const int ks = j % L::kKS, vs = j % L::kVS;
      const int k0 = w.k0(j);
      uint8_t* sK = sm + L::kK + ks * L::kTileBytes;
      uint8_t* sV = sm + L::kV + vs * L::kTileBytes;
      check(k0 >= 0 && k0 < s.T && hk < s.Hkv, err, 1002);
      if (j >= L::kKS && !mbar_wait(&bar[kKEmpty + ks], ((j / L::kKS) - 1) & 1, err, 101)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bar[kKFull + ks], L::kTileBytes);
        for (int a = 0; a < D / 64; ++a) tma_load_3d(sK + a * 16384, &mK, &bar[kKFull + ks], a * 64, hk, k0);
      }
      k_issued = j + 1;
      if (j >= L::kVS && !mbar_wait(&bar[kVEmpty + vs], ((j / L::kVS) - 1) & 1, err, 102)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bar[kVFull + vs], L::kTileBytes);
        for (int a = 0; a < D / 64; ++a) tma_load_3d(sV + a * 16384, &mV, &bar[kVFull + vs], a * 64, hk, k0);
      }
      v_issued = j + 1;
    }
    if (lane == 0) steps.put(0, v_issued);
    // Before the CTA can exit, every copy this warp issued must have landed
    // (the consumers may have stopped early on an error).
    for (int j = (k_issued > L::kKS ? k_issued - L::kKS : 0); j < k_issued; ++j)
      mbar_wait(&bar[kKFull + j % L::kKS], (j / L::kKS) & 1, err, 103);
    for (int j = (v_issued > L::kVS ? v_issued - L::kVS : 0); j < v_issued; ++j)
      mbar_wait(&bar[kVFull + j % L::kVS], (j / L::kVS) & 1, err, 104);
    mbar_wait(&bar[kQFull], 0, err, 105);
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idO = idesc_bf16(128, D, false, true);
    bool ok = mbar_wait(&bar[kQFull], 0, err, 201);
    // S_x(j) = Q_x K_j^T; the K stage is released after the last head's product
    auto issue_s = [&](int j, int x) -> bool {
      const int ks = j % L::kKS;
      if (x == 0 && !mbar_wait(&bar[kKFull + ks], (j / L::kKS) & 1, err, 202)) return false;
      tc_fence_after();
      const uint32_t sQ = smem_u32(sm + L::kQ + x * L::kTileBytes);
      const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        if (elect_one())
          mma_ss(tmem + col_s(x), desc_kmajor_sw128(sQ + off), desc_kmajor_sw128(sK + off), idS, kk > 0 ? 1u : 0u);
      }
      if (elect_one()) mma_commit(&bar[kSFull + x]);
      if (x == nheads - 1 && elect_one()) mma_commit(&bar[kKEmpty + ks]);
      return true;
    };
    for (int x = 0; ok && x < nheads; ++x) ok = issue_s(0, x);
    int done = 0;
    for (int j = 0; ok && j < n; ++j) {
      const int vs = j % L::kVS;
      const uint32_t sV = smem_u32(sm + L::kV + vs * L::kTileBytes);
      for (int x = 0; ok && x < nheads; ++x) {
        if (!mbar_wait(&bar[kPFull + x], j & 1, err, 204)) { ok = false; break; }
        if (x == 0 && !mbar_wait(&bar[kVFull + vs], (j / L::kVS) & 1, err, 205)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          if (elect_one())
            mma_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8, desc_mnmajor_sw128(sV + kk * 2048, 16384), idO,
                   (j > 0 || kk > 0) ? 1u : 0u);
        if (x == nheads - 1 && elect_one()) mma_commit(&bar[kVEmpty + vs]);
        if (j + 1 < n) {
          // overwrites this head's S/P block; in issue order after the PV that reads P
          if (!issue_s(j + 1, x)) { ok = false; break; }
        } else if (elect_one()) {
          mma_commit(&bar[kODone + x]);
        }
      }
      if (ok) done = j + 1;
    }
    if (lane == 0) steps.put(1, done);
  } else if (warp / 4 < nheads) {
    // ---------------------------------------------------------------- softmax
    const int x = warp >> 2;  // head of this warpgroup
    const int h = h0 + x;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(x);
    const uint32_t tO = tmem + lane_off + col_o(x);
    const float c = s.scale_log2;
    float m_use = -INFINITY;
    float l = 0.f;   // sum of the fp32 probabilities (for the LSE)
    float lr = 0.f;  // sum of their bf16 roundings (normalises O)
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(&bar[kSFull + x], j & 1, err, 301)) { ok = false; break; }
      tc_fence_after();
      const int mk = w.mask_kind(j);
      const int lim = (mk == 2) ? w.key_limit(j) : (mk == 1 ? row + 1 : kTile);  // columns >= lim are masked
      const float mt = (mk == 0) ? row_max<false>(tS, lim) : row_max<true>(tS, lim);
      const float m_cand = mt * c;
      // Keep the running maximum unless it grows by more than 2^8: the final
      // normalisation is exact for any reference value, and skipping the
      // rescale leaves O in TMEM untouched on most tiles.
      const bool resc = m_cand > m_use + 8.f;
      const float m_new = resc ? m_cand : m_use;
      const float alpha = resc ? ex2(m_use - m_new) : 1.f;
      const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
      // O is stable here: the previous PV of this head completed before these scores did.
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int ci = 0; ci < D / 32; ++ci) {
          uint32_t r[32];
          tmem_ld32(tO + ci * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + ci * 32, r);
        }
      }
      const float2 rs = (mk == 0) ? row_exp<false>(tS, lim, c, m_sub) : row_exp<true>(tS, lim, c, m_sub);
      l = l * alpha + rs.x;
      lr = lr * alpha + rs.y;
      m_use = m_new;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();  // every lane's P (and rescaled O) is stored and fenced
      if (lane == 0) mbar_arrive(&bar[kPFull + x]);
      if (row == 0) steps.put(2 + x, j + 1);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&bar[kODone + x], 0, err, 303);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int q = w.q0 + row;
      const bool valid = q < w.q_end;
      const float inv_l = 1.f / lr;
      uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(q) * s.Hq + h) * D);
#pragma unroll
      for (int ci = 0; ci < D / 32; ++ci) {
        uint32_t r[32];
        tmem_ld32(tO + ci * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
        if (valid && check(q >= 0 && q < s.T && h < s.Hq, err, 1003)) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[ci * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (valid && check(q >= 0 && q < s.T && h < s.Hq, err, 1003))
        lse[static_cast<size_t>(h) * s.T + q] = (m_use + log2f(l)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 256) steps.verify(n, err, 1004);
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
  const unsigned grid = static_cast<unsigned>(s.num_items) * static_cast<unsigned>(fwd_head_slots(s.Hq, s.group));
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
