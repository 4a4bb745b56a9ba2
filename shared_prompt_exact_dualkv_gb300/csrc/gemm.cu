// bf16 GEMMs of the packed decoder layer on the tcgen05 tensor cores.
//
// The layer's projections and MLP are plain per-token matrix products on the
// packed P + N*R rows (DualKV abstract page: the repacking extends the token
// saving to the entire model).  Three row-major forms cover forward, dX and dW:
//   kind 0  Y[M,N]  (+)= A[M,K] . B[N,K]^T    (activations x weights^T)
//   kind 1  Y[M,N]   = A[M,K] . B[K,N]        (output grads x weights)
//   kind 2  Y[M,N]   = A[K,M]^T . B[K,N]      (weight grads, fp32 out)
// bf16 operands, fp32 accumulation in TMEM, bf16 (kinds 0, 1) or fp32
// (kind 2) results.  With `accumulate` the bf16 result is added to what Y
// holds (the residual add of the layer).
//
// Persistent kernel, one CTA per SM, output tiles of BM x 256 walked with a
// stride of the grid.  Warp 0 copies A/B k-blocks (64 deep) with TMA into a
// ring of stages; warp 1 owns TMEM and issues tcgen05.mma (M=128, N=256,
// K=16).  With BM = 128 the products go into one of two 256-column
// accumulators and warps 2-5 drain the other (TMEM -> registers -> global)
// while the next tile is computed; with BM = 256 two products per k-step
// (the two 128-row halves of A against one B block) fill both accumulators
// and warps 2-9 drain them together.
// Every wait is bounded (an expired wait records a timeout and the kernel
// returns).
#include <cuda_bf16.h>

#include "checks.cuh"
#include "layer_kernels.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace dkv {
namespace {

constexpr int kBN = 256, kBK = 64;

// Tile shapes: BM = 128 rows keeps two 256-column accumulators in TMEM, so
// the epilogue of one tile overlaps the next tile's products; BM = 256 rows
// uses both accumulators for one tile (two M = 128 products share every B
// k-block), which halves the B bytes each SM copies per product flop.
template <int BM>
struct GemmCfg {
  static constexpr int kStages = BM == 128 ? 4 : 3;
  static constexpr int kBufs = BM == 128 ? 2 : 1;   // accumulators per tile in flight
  static constexpr int kEpiWarps = BM == 128 ? 4 : 8;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kABytes = BM * kBK * 2;
  static constexpr int kBBytes = kBN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers, TMEM slot, alignment slack
};

// barriers: full[stage], empty[stage], acc_full[buf], acc_empty[buf]
constexpr int kFull = 0, kEmpty = 4, kAccFull = 8, kAccEmpty = 10;

struct GemmArgs {
  void* y;
  int32_t M, N, K;
  int64_t ldy;          // elements between rows of Y
  int32_t accumulate;   // kinds 0/1: Y += result
};

template <int KIND, int BM>
__global__ void __launch_bounds__(GemmCfg<BM>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                const __grid_constant__ GemmArgs g, unsigned int* err) {
  using C = GemmCfg<BM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kBarOff + 128);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (g.M + BM - 1) / BM;
  const int tiles_n = (g.N + kBN - 1) / kBN;
  const int tiles = tiles_m * tiles_n;
  const int kblocks = (g.K + kBK - 1) / kBK;

  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bar[kFull + i], 1);
      mbar_init(&bar[kEmpty + i], 1);
    }
    for (int i = 0; i < C::kBufs; ++i) {
      mbar_init(&bar[kAccFull + i], 1);
      mbar_init(&bar[kAccEmpty + i], 32 * C::kEpiWarps);
    }
    fence_mbar_init();
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    int it = 0;  // k-blocks issued over all tiles of this CTA
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
      const int m0 = (t / tiles_n) * BM, n0 = (t % tiles_n) * kBN;
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int st = it % C::kStages;
        if (it >= C::kStages && !mbar_wait(&bar[kEmpty + st], ((it / C::kStages) - 1) & 1, err, 1501)) {
          ok = false;
          break;
        }
        uint8_t* sA = sm + st * C::kStageBytes;
        uint8_t* sB = sA + C::kABytes;
        const int k0 = kb * kBK;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bar[kFull + st], C::kStageBytes);
          if (KIND == 2) {
            // A[K,M]: BM/64 blocks of 64 M columns x 64 K rows
            for (int a = 0; a < BM / 64; ++a) tma_load_2d(sA + a * 8192, &mA, &bar[kFull + st], m0 + a * 64, k0);
          } else {
            tma_load_2d(sA, &mA, &bar[kFull + st], k0, m0);
          }
          if (KIND == 0) {
            tma_load_2d(sB, &mB, &bar[kFull + st], k0, n0);
          } else {
            // B[K,N]: four blocks of 64 N columns x 64 K rows
            for (int a = 0; a < kBN / 64; ++a) tma_load_2d(sB + a * 8192, &mB, &bar[kFull + st], n0 + a * 64, k0);
          }
        }
        __syncwarp();
      }
    }
    // every copy issued must land before the CTA exits
    for (int i = (it > C::kStages ? it - C::kStages : 0); i < it; ++i)
      mbar_wait(&bar[kFull + i % C::kStages], (i / C::kStages) & 1, err, 1502);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(128, kBN, KIND == 2, KIND >= 1);
    int it = 0, local = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++local) {
      const int buf = local % C::kBufs, use = local / C::kBufs;
      // the epilogue has drained this accumulator (its previous tile)
      if (use >= 1 && !mbar_wait(&bar[kAccEmpty + buf], (use - 1) & 1, err, 1503)) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * kBN;  // BM = 256: both halves, columns [0, 512)
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int st = it % C::kStages;
        if (!mbar_wait(&bar[kFull + st], (it / C::kStages) & 1, err, 1504)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = smem_u32(sm + st * C::kStageBytes);
        const uint32_t sB = sA + C::kABytes;
#pragma unroll
        for (int hm = 0; hm < BM / 128; ++hm) {
          // rows 128*hm.. of the A tile into columns 256*hm.. of TMEM
          const uint32_t sAh = sA + hm * 16384;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t da =
                KIND == 2 ? desc_mnmajor_sw128(sAh + kk * 2048, 8192) : desc_kmajor_sw128(sAh + kk * 32);
            const uint64_t db =
                KIND == 0 ? desc_kmajor_sw128(sB + kk * 32) : desc_mnmajor_sw128(sB + kk * 2048, 8192);
            if (elect_one()) mma_ss(acc + hm * kBN, da, db, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (elect_one()) mma_commit(&bar[kEmpty + st]);
        __syncwarp();
      }
      if (ok && elect_one()) mma_commit(&bar[kAccFull + buf]);
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int part = (warp - 2) / 4;       // BM = 256: which 128-row half
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    int local = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
      const int buf = local % C::kBufs, use = local / C::kBufs;
      const int m0 = (t / tiles_n) * BM, n0 = (t % tiles_n) * kBN;
      if (!mbar_wait(&bar[kAccFull + buf], use & 1, err, 1505)) break;
      tc_fence_after();
      const int row = m0 + part * 128 + quarter * 32 + lane;
      const uint32_t col0 = (BM == 128 ? buf : part) * kBN;
      const bool row_ok = row < g.M && check(row >= 0, err, 1506);
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + col0 + c * 32, r);
        tmem_ld_wait();
        const int col = n0 + c * 32;
        if (!row_ok || col >= g.N) {
          // nothing of this chunk lies inside Y
        } else if (KIND == 2) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(g.y) + row * g.ldy + col);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (col + 4 * v < g.N)
              dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.y) + row * g.ldy + col);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (col + 8 * v >= g.N) continue;
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[8 * v + i]);
            if (g.accumulate) {
              const uint4 old = dst[v];
              const __nv_bfloat162* ob = reinterpret_cast<const __nv_bfloat162*>(&old);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 o2 = __bfloat1622float2(ob[i]);
                f[2 * i] += o2.x;
                f[2 * i + 1] += o2.y;
              }
            }
            dst[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar[kAccEmpty + buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// Tile height for a product: 256 rows when the output has enough 256 x 256
// tiles to fill every SM at least twice, else 128 (more, smaller tiles).
int tile_rows(int64_t M, int64_t N) {
  const int64_t t256 = ((M + 255) / 256) * ((N + kBN - 1) / kBN);
  return t256 >= 2 * sm_count() ? 256 : 128;
}

template <int KIND, int BM>
cudaError_t launch_kind(const CUtensorMap& mA, const CUtensorMap& mB, const GemmArgs& a, unsigned int* err,
                        cudaStream_t stream) {
  using C = GemmCfg<BM>;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_kernel<KIND, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + kBN - 1) / kBN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  gemm_kernel<KIND, BM><<<grid, C::kThreads, C::kSmemBytes, stream>>>(mA, mB, a, err);
  return cudaGetLastError();
}

}  // namespace

// Row-major bf16 matrix [rows, cols] (cols contiguous) as a 2-D tensor map
// with a box of 64 columns (128 B, 128-byte swizzle) x box_rows.
static bool map_2d(CUtensorMap* m, const void* p, int64_t rows, int64_t cols, int box_rows) {
  return make_map_2d(m, p, rows, cols, 64, box_rows);
}

cudaError_t gemm_xwT(int64_t M, int N, int K, const void* X, const void* W, void* Y, bool accumulate,
                     unsigned int* err, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int bm = tile_rows(M, N);
  CUtensorMap mA, mB;
  if (!map_2d(&mA, X, M, K, bm) || !map_2d(&mB, W, N, K, kBN)) return cudaErrorInvalidValue;
  GemmArgs a{Y, static_cast<int32_t>(M), N, K, N, accumulate ? 1 : 0};
  return bm == 256 ? launch_kind<0, 256>(mA, mB, a, err, stream) : launch_kind<0, 128>(mA, mB, a, err, stream);
}

cudaError_t gemm_dyW(int64_t M, int N, int K, const void* dY, const void* W, void* dX, unsigned int* err,
                     cudaStream_t stream) {
  // dX[M, N] = dY[M, K] . W[K, N]
  if (M == 0) return cudaSuccess;
  const int bm = tile_rows(M, N);
  CUtensorMap mA, mB;
  if (!map_2d(&mA, dY, M, K, bm) || !map_2d(&mB, W, K, N, 64)) return cudaErrorInvalidValue;
  GemmArgs a{dX, static_cast<int32_t>(M), N, K, N, 0};
  return bm == 256 ? launch_kind<1, 256>(mA, mB, a, err, stream) : launch_kind<1, 128>(mA, mB, a, err, stream);
}

cudaError_t gemm_dW(int M, int N, int64_t K, const void* dY, const void* X, float* dW, unsigned int* err,
                    cudaStream_t stream) {
  // dW[M, N] = dY[K, M]^T . X[K, N]
  if (K == 0) return cudaMemsetAsync(dW, 0, size_t(M) * N * 4, stream);
  const int bm = tile_rows(M, N);
  CUtensorMap mA, mB;
  if (!map_2d(&mA, dY, K, M, 64) || !map_2d(&mB, X, K, N, 64)) return cudaErrorInvalidValue;
  GemmArgs a{dW, M, N, static_cast<int32_t>(K), N, 0};
  return bm == 256 ? launch_kind<2, 256>(mA, mB, a, err, stream) : launch_kind<2, 128>(mA, mB, a, err, stream);
}

}  // namespace dkv
