// Host-side TMA tensor-map encoding.  The driver entry point is fetched through
// the runtime, so the library needs no link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace dkv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// The encoder is a driver call and needs a current context on the calling
// thread.  A thread whose first CUDA work this is (an autograd worker thread,
// say) has none until a runtime call binds the device's primary context,
// which cudaSetDevice does.
inline bool bind_primary_context() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
}

// The driver's result for the calling thread's last rejected tensor map
// (-1: no encoder, no context or invalid arguments).
inline int& last_map_result() {
  static thread_local int r = 0;
  return r;
}

inline bool encode_failed(int r) {
  last_map_result() = r;
  return false;
}

// Tensor map over a row-major [T, H, d] bf16 tensor (token, head, feature).
// One box is 64 features (128 B, one swizzle row) x 1 head x `box_rows`
// tokens, landing in shared memory as `box_rows` 128-byte rows with the
// 128-byte swizzle.  Tokens past T read as zero.
// Returns false if the driver rejects the map.
inline bool make_map_thd(CUtensorMap* m, const void* base, int64_t T, int H, int d, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || !bind_primary_context()) return encode_failed(-1);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2};
  cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS || encode_failed(static_cast<int>(r));
}

// Tensor map over a row-major [rows, cols] bf16 matrix (cols contiguous, a
// multiple of 8).  One box is box_cols (64: 128 B, one swizzle row) x
// box_rows, landing as box_rows 128-byte rows with the 128-byte swizzle.
// Elements past either extent read as zero.
inline bool make_map_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || rows < 1 || cols < 1 || cols % 8 != 0 || !bind_primary_context()) return encode_failed(-1);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS || encode_failed(static_cast<int>(r));
}

}  // namespace dkv
