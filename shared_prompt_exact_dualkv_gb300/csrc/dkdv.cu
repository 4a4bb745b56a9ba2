// dK/dV kernel of the backward pass.
//
// One CTA owns one 128-row key tile of one kv-head (and, for prompt key
// tiles, one chunk of the N sequences).  It loops over every query tile that
// sees those keys, for all q-heads of the kv-head's group (GQA):
//   * a response key tile of sequence i: the later query tiles of response i,
//     from the last one down to the diagonal (masked causally), so the key
//     tiles of one response, which run together, read the same query tile
//     at about the same time;
//   * a prompt key tile: the prompt's own later query tiles (split 0 only,
//     causal) and every query tile of the responses in its chunk (no mask):
//     the prompt keys are shared by all N sequences (DualKV research-map page,
//     "Approach"; abstract: the prompt is processed once).
// Per query tile, with keys on TMEM lanes (FlashAttention-2 style backward):
//   S^T = K Q^T, P^T = exp(scale*S^T - LSE), dP^T = V dO^T,
//   dS^T = P^T * (dP^T - D), dV += P^T dO, dK += dS^T Q;  dK *= scale.
// Response key rows are written as bf16.  Prompt key rows are fp32 partial
// sums over this CTA's sequences; they are added with fp32 atomics into one
// accumulator (research-map page, "Approach") or, in deterministic mode,
// stored per split and summed in a fixed order by the reduce kernel.
//
// Warp roles (320 threads): warps 0-7 elementwise -- warp w handles key rows
// 32*(w%4) .. +31 (its TMEM lane quarter) and query columns 64*(w/4) .. +63,
// so each row is split over two warps and every SM sub-partition runs two
// elementwise warps; warp 8 producer (TMA for Q/dO tiles; its 32 lanes stage
// the LSE and D vectors of each query tile); warp 9 TMEM allocator + MMA issuer.
// TMEM columns: S^T [0,128); dP^T [128,256); dV [256,256+D); dK [384,384+D).
// Each half writes its bf16 P^T over the S^T columns it has already read
// (query half h -> columns [64h, 64h+32)), and likewise dS^T over dP^T, so
// the two halves never touch each other's unread columns.
#include <cuda_bf16.h>

#include "checks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {
namespace {

// FQ: the variant that also computes dQ (the dS tile then lives in shared
// memory).  Its layout has no alignment slack: it only fits with the
// dynamic shared memory starting 1024-byte aligned, which the kernel checks.
template <int D, bool FQ>
struct DkdvLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kdO = kQ + kStages * kTileBytes;
  static constexpr int kdS = kdO + kStages * kTileBytes;    // FQ: dS^T [2 query halves][128 keys][128 B]
  static constexpr int kVec = kdS + (FQ ? kTile * kTile * 2 : 0);  // per stage: lse2[128], D[128] floats
  static constexpr int kBar = kVec + kStages * 1024;
  static constexpr int kSlack = FQ ? 0 : 1024;
  static constexpr int kBytes = kBar + 256 + kSlack;
};

enum DkdvBar {
  kKVFull = 0,
  kQFull = 1,    // + stage
  kQEmpty = 3,   // + stage
  kSFull = 5,
  kdPFull = 6,
  kPReady = 7,
  kdSReady = 8,
  kAccDone = 9,
  kdQFull = 10,  // FQ: this tile's dQ product is in TMEM (over the dP^T columns)
  kdQFree = 11,  // FQ: the elementwise warps have read it out
  kNumDkdvBars = 12
};

constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 384;
// Each key row's 128 query columns are split over kColGroups elementwise
// warps (the same TMEM lane quarter, different columns); the groups need no
// exchange, the work being elementwise.
constexpr int kColGroups = 2;
constexpr int kCols = kTile / kColGroups;        // query columns per elementwise thread
constexpr int kEwWarps = 4 * kColGroups;
constexpr int kEwThreads = 32 * kEwWarps;
constexpr int kThreads = kEwThreads + 64;        // + the copy producer and the MMA issuer
constexpr int kProducerWarp = kEwWarps, kMmaWarp = kEwWarps + 1;

// TMEM column offset of the K=16 slice kk of a bf16 operand that each column
// group g stored (packed two per column) at the start of its own range,
// columns [g*kCols, g*kCols + kCols/2).
__device__ __forceinline__ uint32_t split_col(int kk) {
  return (16 * kk / kCols) * kCols + (16 * kk % kCols) / 2;
}

// The query tiles seen by one key-tile item, as "runs" of consecutive tiles
// of one segment; the walk repeats the runs for each q-head of the group.
struct QRuns {
  int32_t seg, j, split, nP, has_prompt, seq_lo, num_runs, per_head, group, hk;
  int32_t k0, k_end;     // key rows of the item
  int32_t prompt_item;   // 1 for a prompt key tile
  int32_t acc0;          // prompt key tile: accumulator row of its first key

  __device__ __forceinline__ void init(const Sched& s, uint32_t item, int32_t kvh) {
    seg = static_cast<int32_t>(item_seg(item));
    j = static_cast<int32_t>(item_tile(item));
    split = static_cast<int32_t>(item_split(item));
    group = s.group;
    hk = kvh;
    per_head = 0;
    k0 = s.off[seg] + j * kTile;
    k_end = s.off[seg + 1];
    prompt_item = s.prompt_of(seg) == seg ? 1 : 0;
    if (prompt_item) {
      // the group's responses are the segments right after its prompt
      const int32_t ng = s.responses_of(seg);
      nP = s.seg_tiles(seg);
      has_prompt = split == 0 ? 1 : 0;
      seq_lo = seg + 1 + (split * ng) / s.num_splits;
      const int seq_hi = seg + 1 + ((split + 1) * ng) / s.num_splits;
      num_runs = has_prompt + (seq_hi - seq_lo);
      // the prompt's own query tiles j..nP-1 (causal), within the part taken
      if (has_prompt) per_head += max(0, min(nP, s.pq_hi) - max(j, s.pq_lo));
      for (int i = seq_lo; i < seq_hi; ++i) per_head += s.seg_tiles(i);
      acc0 = s.acc_row[seg] + j * kTile;
    } else {
      nP = 0;
      has_prompt = 0;
      seq_lo = seg;
      num_runs = 1;
      per_head = s.seg_tiles(seg) - j;
      acc0 = 0;
    }
  }
};

// Walk order of one key-tile item, per q-head of the group.  A prompt key
// tile: the query tiles of the responses in its chunk first, ascending, then
// (split 0) the prompt's own query tiles, descending from the last to the key
// tile's diagonal.  A response key tile: its response's query tiles,
// descending from the last to the diagonal.  The key tiles whose CTAs run
// together (one group's prompt tiles, or one response's tiles) thus work on
// the same query tiles at about the same time, and L2 serves those tiles
// (and, with dQ fused, takes their dQ reductions) for all of them.
struct QIter {
  int32_t hh, r, t, step, t_stop;   // t runs from its first tile by `step` until it reaches t_stop
  int32_t q_first, seg_end;
  int32_t diag_t;   // the query tile on the key tile's diagonal (-1: none in this run)

  __device__ __forceinline__ int32_t resp_runs(const QRuns& R) const { return R.num_runs - R.has_prompt; }

  __device__ __forceinline__ void load_run(const Sched& s, const QRuns& R) {
    if (r < resp_runs(R)) {
      const int i = R.seq_lo + r;
      q_first = s.off[i];
      seg_end = s.off[i + 1];
      if (R.prompt_item) {
        t = 0;
        t_stop = s.seg_tiles(i);
        step = 1;
        diag_t = -1;
      } else {
        t = s.seg_tiles(i) - 1;
        t_stop = R.j - 1;
        step = -1;
        diag_t = R.j;
      }
    } else {
      q_first = s.off[R.seg];
      t = min(R.nP, s.pq_hi) - 1;
      t_stop = max(R.j, s.pq_lo) - 1;
      step = -1;
      seg_end = s.off[R.seg + 1];
      diag_t = R.j;
    }
  }
  __device__ __forceinline__ bool run_done() const { return step > 0 ? t >= t_stop : t <= t_stop; }
  __device__ __forceinline__ void skip_empty(const Sched& s, const QRuns& R) {
    while (run_done()) {
      if (++r == R.num_runs) {
        r = 0;
        ++hh;
      }
      load_run(s, R);
    }
  }
  // Position on the first query tile (the item must have per_head > 0).
  __device__ __forceinline__ void start(const Sched& s, const QRuns& R) {
    hh = 0;
    r = 0;
    load_run(s, R);
    skip_empty(s, R);
  }
  __device__ __forceinline__ void next(const Sched& s, const QRuns& R) {
    t += step;
    skip_empty(s, R);
  }
  __device__ __forceinline__ int32_t q0() const { return q_first + t * kTile; }
  __device__ __forceinline__ bool diag() const { return t == diag_t; }
  __device__ __forceinline__ int32_t head(const QRuns& R) const { return R.hk * R.group + hh; }
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// TMEM load of N (16, 32 or a multiple of 32) consecutive columns of this
// warp's lanes, and store of N packed columns (16 or 32).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  static_assert(N == 16 || N % 32 == 0, "TMEM load width");
  if constexpr (N == 16) {
    tmem_ld16(taddr, r);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32(taddr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(r + c * 32));
  }
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  static_assert(N == 16 || N == 32, "TMEM store width");
  if constexpr (N == 16) {
    tmem_st16(taddr, r);
  } else {
    tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(r));
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// dq_acc (FQ only): fp32 dQ accumulator [Hq][D/4][T][4] (unscaled); each
// tile's dQ = dS K is added to it with fp32 vector reductions.
template <int D, bool FQ>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ Sched s, const __grid_constant__ CUtensorMap mQ,
                const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const __grid_constant__ CUtensorMap mdO, const float* __restrict__ lse,
                const float* __restrict__ Dvec, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                float* __restrict__ acc_k, float* __restrict__ acc_v, float* __restrict__ dq_acc, int deterministic,
                unsigned int* err) {
  using L = DkdvLayout<D, FQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = FQ ? smem_raw
                  : reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (FQ && (smem_u32(smem_raw) & 1023u) != 0) {
    // the layout needs a 1024-byte aligned base (every thread takes this exit)
    if (threadIdx.x == 0) record_error(err, kDevErrCheck, 1107);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kBar + 128);
  const RoleSteps steps{reinterpret_cast<int32_t*>(sm + L::kBar + 160)};  // checks build only
  float* vec = reinterpret_cast<float*>(sm + L::kVec);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t item = s.items[blockIdx.x / s.Hkv];
  const int hk = blockIdx.x % s.Hkv;
  QRuns R;
  R.init(s, item, hk);
  const int n = R.per_head * R.group;

  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == kEwThreads) {
    mbar_init(&bar[kKVFull], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kQFull + i], 2);
      mbar_init(&bar[kQEmpty + i], 1);
    }
    mbar_init(&bar[kSFull], 1);
    mbar_init(&bar[kdPFull], 1);
    mbar_init(&bar[kPReady], kEwThreads);
    mbar_init(&bar[kdSReady], kEwThreads);
    mbar_init(&bar[kAccDone], 1);
    mbar_init(&bar[kdQFull], 1);
    mbar_init(&bar[kdQFree], kEwThreads);
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

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (n > 0) {
      // (an out-of-range tile copy would only read zeros; the checks record it)
      check(R.k0 >= 0 && R.k0 < s.T && hk < s.Hkv, err, 1101);
      if (elect_one()) {
        mbar_arrive_expect_tx(&bar[kKVFull], 2 * L::kTileBytes);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(sm + L::kK + a * 16384, &mK, &bar[kKVFull], a * 64, hk, R.k0);
          tma_load_3d(sm + L::kV + a * 16384, &mV, &bar[kKVFull], a * 64, hk, R.k0);
        }
      }
      // Each query tile's LSE/D values are read into registers one tile ahead,
      // so their global-load latency overlaps the previous tile; a stage's
      // full barrier takes two arrivals: the copy's expect-tx and "vectors stored".
      QIter it;
      it.start(s, R);
      float l2[4], dd[4];
      auto load_vec = [&](const QIter& t) {
        const int h = t.head(R);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = t.q0() + lane * 4 + u;
          l2[u] = INFINITY;
          dd[u] = 0.f;
          if (q < t.seg_end && check_index(static_cast<int64_t>(h) * s.T + q, static_cast<int64_t>(s.Hq) * s.T, err, 1103)) {
            l2[u] = lse[static_cast<size_t>(h) * s.T + q] * 1.4426950408889634f;
            dd[u] = Dvec[static_cast<size_t>(h) * s.T + q];
          }
        }
      };
      load_vec(it);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i & 1;
        if (i >= 2 && !mbar_wait(&bar[kQEmpty + st], ((i >> 1) - 1) & 1, err, 701)) break;
        check(it.q0() >= 0 && it.q0() < s.T && it.head(R) < s.Hq, err, 1102);
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kQFull + st], 2 * L::kTileBytes);
          for (int a = 0; a < D / 64; ++a) {
            tma_load_3d(sm + L::kQ + st * L::kTileBytes + a * 16384, &mQ, &bar[kQFull + st], a * 64, it.head(R), it.q0());
            tma_load_3d(sm + L::kdO + st * L::kTileBytes + a * 16384, &mdO, &bar[kQFull + st], a * 64, it.head(R), it.q0());
          }
        }
        issued = i + 1;
        if (lane == 0) steps.put(0, issued);
        float* vl = vec + st * 256;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          vl[lane * 4 + u] = l2[u];
          vl[128 + lane * 4 + u] = dd[u];
        }
        __syncwarp();
        if (elect_one()) mbar_arrive(&bar[kQFull + st]);
        __syncwarp();
        if (i + 1 < n) {
          it.next(s, R);
          load_vec(it);
        }
      }
      // Before the CTA can exit, every copy this warp issued must have landed
      // (the consumers may have stopped early on an error).
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        mbar_wait(&bar[kQFull + (i & 1)], (i >> 1) & 1, err, 702);
      mbar_wait(&bar[kKVFull], 0, err, 703);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // The warp runs the loop converged (warp-uniform control flow and
    // descriptors); one elected lane issues each MMA and commit.
    if (n > 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idG = idesc_bf16(128, D, false, true);
      const uint32_t sK = smem_u32(sm + L::kK);
      const uint32_t sV = smem_u32(sm + L::kV);
      bool ok = mbar_wait(&bar[kKVFull], 0, err, 801);
      auto issue_s = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait(&bar[kQFull + st], (i >> 1) & 1, err, 802)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_u32(sm + L::kQ + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (elect_one()) mma_ss(tmem + kColS, desc_kmajor_sw128(sK + off), desc_kmajor_sw128(sQ + off), idSS, kk > 0 ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kSFull]);
        return true;
      };
      auto issue_dp = [&](int i) {
        const int st = i & 1;
        const uint32_t sdO = smem_u32(sm + L::kdO + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (elect_one()) mma_ss(tmem + kColdP, desc_kmajor_sw128(sV + off), desc_kmajor_sw128(sdO + off), idSS, kk > 0 ? 1u : 0u);
        }
        if (elect_one()) mma_commit(&bar[kdPFull]);
      };
      if (ok) {
        ok = issue_s(0);
        if (ok) issue_dp(0);
      }
      for (int i = 0; ok && i < n; ++i) {
        const int st = i & 1;
        // dV += P^T dO  (P^T read from TMEM columns [0,32) and [64,96))
        if (!mbar_wait(&bar[kPReady], i & 1, err, 803)) break;
        tc_fence_after();
        const uint32_t sdO = smem_u32(sm + L::kdO + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          if (elect_one()) mma_ts(tmem + kColdV, tmem + kColS + split_col(kk), desc_mnmajor_sw128(sdO + kk * 2048, 16384), idG,
                 (i > 0 || kk > 0) ? 1u : 0u);
        // the next S^T may overwrite P^T: it is issued after the dV product
        if (i + 1 < n && !issue_s(i + 1)) break;
        if (!mbar_wait(&bar[kdSReady], i & 1, err, 804)) break;
        tc_fence_after();
        const uint32_t sQ = smem_u32(sm + L::kQ + st * L::kTileBytes);
        if (!FQ) {
          // dK += dS^T Q  (dS^T read from TMEM columns [128,160) and [192,224))
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            if (elect_one()) mma_ts(tmem + kColdK, tmem + kColdP + split_col(kk), desc_mnmajor_sw128(sQ + kk * 2048, 16384), idG,
                   (i > 0 || kk > 0) ? 1u : 0u);
          if (elect_one()) mma_commit(&bar[kQEmpty + st]);
          if (i + 1 < n) issue_dp(i + 1);
        } else {
          // dK += dS^T Q with dS^T from shared memory (keys x queries, K-major), then
          // dQ = dS K into the dP^T columns, which the elementwise warps have read:
          // A = the same tile read queries-major, B = K read d-major.
          constexpr uint32_t idQ = idesc_bf16(128, D, true, true);
          const uint32_t sdS = smem_u32(sm + L::kdS);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            if (elect_one()) mma_ss(tmem + kColdK, desc_kmajor_sw128(sdS + off), desc_mnmajor_sw128(sQ + kk * 2048, 16384),
                                    idG, (i > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            if (elect_one()) mma_ss(tmem + kColdP, desc_mnmajor_sw128(sdS + kk * 2048, 16384),
                                    desc_mnmajor_sw128(sK + kk * 2048, 16384), idQ, kk > 0 ? 1u : 0u);
          if (elect_one()) mma_commit(&bar[kQEmpty + st]);
          if (elect_one()) mma_commit(&bar[kdQFull]);
          // the next dP^T goes where this dQ is: wait until it has been read out
          if (i + 1 < n) {
            if (!mbar_wait(&bar[kdQFree], i & 1, err, 805)) break;
            tc_fence_after();
            issue_dp(i + 1);
          }
        }
        if (lane == 0) steps.put(1, i + 1);
      }
      if (elect_one()) mma_commit(&bar[kAccDone]);
    }
  } else {
    // ---------------------------------------------------------------- elementwise
    constexpr int kDq = D / kColGroups;          // dQ / dK / dV columns per thread
    constexpr int kCh = kDq < 32 ? kDq : 32;     // columns per TMEM load of those
    const int quarter = warp & 3;
    const int grp = warp >> 2;                   // column group
    const int row = quarter * 32 + lane;
    const int cb = grp * kCols;  // first query column of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    const bool key_in = R.k0 + row < R.k_end;
    bool ok = n > 0;
    if (ok) {
      QIter it;
      it.start(s, R);
      for (int i = 0; i < n; ++i, (i < n ? it.next(s, R) : void())) {
        const int st = i & 1;
        const float* vl = vec + st * 256 + cb;
        if (!mbar_wait(&bar[kQFull + st], (i >> 1) & 1, err, 901)) { ok = false; break; }
        if (!mbar_wait(&bar[kSFull], i & 1, err, 902)) { ok = false; break; }
        tc_fence_after();
        float p[kCols];
        {
          uint32_t r[kCols];
          tmem_ld_cols<kCols>(tmem + lane_off + kColS + cb, r);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < kCols; ++u) p[u] = __uint_as_float(r[u]);
        }
#pragma unroll
        for (int u = 0; u < kCols; u += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(vl + u);
          const float2 a0 = fma2(make_float2(p[u], p[u + 1]), make_float2(c, c), make_float2(-l4.x, -l4.y));
          const float2 a1 = fma2(make_float2(p[u + 2], p[u + 3]), make_float2(c, c), make_float2(-l4.z, -l4.w));
          p[u] = ex2(a0.x);
          p[u + 1] = ex2(a0.y);
          p[u + 2] = ex2(a1.x);
          p[u + 3] = ex2(a1.y);
        }
        if (it.diag()) {
#pragma unroll
          for (int u = 0; u < kCols; ++u) p[u] = (cb + u < row) ? 0.f : p[u];
        }
        if (FQ && !key_in) {
          // a key lane past the item's segment (the ragged end of a prompt
          // tile holds the first keys of the next segment) must not reach dQ
#pragma unroll
          for (int u = 0; u < kCols; ++u) p[u] = 0.f;
        }
        {
          uint32_t pk[kCols / 2];
#pragma unroll
          for (int u = 0; u < kCols / 2; ++u) pk[u] = pack_bf16x2(p[2 * u], p[2 * u + 1]);
          tmem_st_cols<kCols / 2>(tmem + lane_off + kColS + cb, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[kPReady]);

        if (!mbar_wait(&bar[kdPFull], i & 1, err, 903)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < kCols / 32; ++ci) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + kColdP + cb + ci * 32, r);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int cc = ci * 32 + 2 * u;
            const float2 d2 = *reinterpret_cast<const float2*>(vl + 128 + cc);
            const float2 t = add2(make_float2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])),
                                  make_float2(-d2.x, -d2.y));
            const float2 ds = mul2(make_float2(p[cc], p[cc + 1]), t);
            pk[u] = pack_bf16x2(ds.x, ds.y);
          }
          if (!FQ) {
            tmem_st16(tmem + lane_off + kColdP + cb + ci * 16, pk);
          } else {
            // row `row` (a key) of its query columns cb.., 128-byte swizzled
            // in the 64-query atom they fall in: the 16-byte chunk j of the
            // row lands at chunk j ^ (row % 8).  The tile's previous contents
            // were last read by the previous dK/dQ products, which completed
            // before the previous drain.
            const uint32_t rowb = smem_u32(sm + L::kdS + (cb / 64) * 16384 + row * 128);
            const int ch0 = (cb % 64) / 8 + ci * 4;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st_shared_v4(rowb + (((ch0 + v) ^ (row & 7)) << 4), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        if (!FQ) {
          tmem_st_wait();
        } else {
          fence_proxy_async_smem();  // the tensor cores read the tile through the async proxy
        }
        tc_fence_before();
        mbar_arrive(&bar[kdSReady]);
        if (FQ) {
          // drain this tile's dQ (query rows on the TMEM lanes, d on the columns)
          // into the fp32 accumulator; the dP^T columns are then free again
          if (!mbar_wait(&bar[kdQFull], i & 1, err, 905)) { ok = false; break; }
          tc_fence_after();
          uint32_t r[kDq];
          tmem_ld_cols<kDq>(tmem + lane_off + kColdP + grp * kDq, r);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bar[kdQFree]);
          const int q = it.q0() + row;
          const int h = it.head(R);
          if (q < it.seg_end && check(q >= 0 && q < s.T && h < s.Hq, err, 1108)) {
            float* base = dq_acc + (static_cast<size_t>(h) * (D / 4) + grp * (kDq / 4)) * s.T * 4 + static_cast<size_t>(q) * 4;
#pragma unroll
            for (int v = 0; v < kDq / 4; ++v)
              red_add_v4(base + static_cast<size_t>(v) * s.T * 4, __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                         __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          }
        }
        if (row == 0 && (grp == 0 || grp == kColGroups - 1)) steps.put(2 + (grp ? 1 : 0), i + 1);
      }
    }
    // ---------------------------------------------------------------- epilogue
    const int k = R.k0 + row;
    const bool valid = k < R.k_end;
    const bool prompt_item = R.prompt_item != 0;
    if (ok) ok = mbar_wait(&bar[kAccDone], 0, err, 904);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) tc_fence_after();
    if (prompt_item) {
      // fp32 partial of this CTA's sequences for prompt key row k, at
      // accumulator row acc0 + row (prompt rows of all groups, packed)
      const size_t base = (static_cast<size_t>(R.acc0 + row) * s.Hkv + hk) * D;
      const size_t slice = static_cast<size_t>(s.acc_rows) * s.Hkv * D;
      float* pk_out = acc_k + (deterministic ? R.split * slice : 0) + base;
      float* pv_out = acc_v + (deterministic ? R.split * slice : 0) + base;
      const bool in_acc = !valid || check(R.acc0 + row < s.acc_rows && R.split < s.num_splits && hk < s.Hkv, err, 1104);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which ? kColdK : kColdV) + grp * kDq;
        const float mul = which ? s.scale : 1.f;
        float* dst = (which ? pk_out : pv_out) + grp * kDq;
#pragma unroll
        for (int ci = 0; ci < kDq / kCh; ++ci) {
          uint32_t r[kCh];
          if (n > 0) {
            tmem_ld_cols<kCh>(tmem + lane_off + col + ci * kCh, r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int u = 0; u < kCh; ++u) r[u] = 0u;
          }
          if (valid && in_acc && (ok || n == 0)) {
#pragma unroll
            for (int u = 0; u < kCh; u += 4) {
              const float a0 = __uint_as_float(r[u]) * mul, a1 = __uint_as_float(r[u + 1]) * mul;
              const float a2 = __uint_as_float(r[u + 2]) * mul, a3 = __uint_as_float(r[u + 3]) * mul;
              if (deterministic)
                *reinterpret_cast<float4*>(dst + ci * kCh + u) = make_float4(a0, a1, a2, a3);
              else if (n > 0)
                red_add_v4(dst + ci * kCh + u, a0, a1, a2, a3);
            }
          }
        }
      }
    } else if (ok) {
      const size_t base = (static_cast<size_t>(k) * s.Hkv + hk) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which ? kColdK : kColdV) + grp * kDq;
        const float mul = which ? s.scale : 1.f;
        uint4* dst = reinterpret_cast<uint4*>((which ? dk : dv) + base + grp * kDq);
#pragma unroll
        for (int ci = 0; ci < kDq / kCh; ++ci) {
          uint32_t r[kCh];
          tmem_ld_cols<kCh>(tmem + lane_off + col + ci * kCh, r);
          tmem_ld_wait();
          uint32_t pk[kCh / 2];
#pragma unroll
          for (int u = 0; u < kCh / 2; ++u)
            pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]) * mul, __uint_as_float(r[2 * u + 1]) * mul);
          if (valid && check(k >= 0 && k < s.T && hk < s.Hkv, err, 1105)) {
#pragma unroll
            for (int v = 0; v < kCh / 8; ++v)
              dst[ci * (kCh / 8) + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == kEwThreads) steps.verify(n, err, 1106);
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool FQ>
cudaError_t launch_dkdv_d(const Sched& s, const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                          const CUtensorMap& mdO, const float* lse, const float* Dvec, void* dk, void* dv,
                          float* acc_k, float* acc_v, float* dq_acc, int deterministic, unsigned int* err,
                          cudaStream_t stream) {
  using L = DkdvLayout<D, FQ>;
  static_assert(L::kBytes <= 232448, "shared memory of one CTA");
  cudaError_t e = cudaFuncSetAttribute(dkdv_kernel<D, FQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(s.num_items) * static_cast<unsigned>(s.Hkv);
  dkdv_kernel<D, FQ><<<grid, kThreads, L::kBytes, stream>>>(s, mQ, mK, mV, mdO, lse, Dvec, static_cast<__nv_bfloat16*>(dk),
                                                       static_cast<__nv_bfloat16*>(dv), acc_k, acc_v, dq_acc,
                                                       deterministic, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dkdv(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                        const CUtensorMap& mdO, const float* lse, const float* Dvec, void* dk, void* dv,
                        float* acc_k, float* acc_v, float* dq_acc, int deterministic, unsigned int* err,
                        cudaStream_t stream) {
  if (s.num_items == 0) return cudaSuccess;
  if (dq_acc != nullptr)
    return d == 64 ? launch_dkdv_d<64, true>(s, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, dq_acc, 0, err, stream)
                   : launch_dkdv_d<128, true>(s, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, dq_acc, 0, err,
                                              stream);
  return d == 64 ? launch_dkdv_d<64, false>(s, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, nullptr,
                                            deterministic, err, stream)
                 : launch_dkdv_d<128, false>(s, mQ, mK, mV, mdO, lse, Dvec, dk, dv, acc_k, acc_v, nullptr,
                                             deterministic, err, stream);
}

}  // namespace dkv
