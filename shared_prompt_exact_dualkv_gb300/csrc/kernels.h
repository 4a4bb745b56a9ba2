// Host-side launchers of the device kernels (one per .cu file).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace dkv {

// Forward: O and LSE for every (query tile, q-head) item of `s`.
cudaError_t launch_fwd(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK,
                       const CUtensorMap& mV, void* out, float* lse, unsigned int* err, cudaStream_t stream);

// Backward preprocess: Dvec[h, t] = sum_c dO[t,h,c] * O[t,h,c] (fp32) for all
// T x Hq rows, and zero `zero_n` floats at `zero_ptr` (the fp32 prompt
// accumulators of the atomic mode; zero_n may be 0).
cudaError_t launch_preprocess(const void* out, const void* dout, float* Dvec, int64_t T, int Hq, int d,
                              float* zero_ptr, size_t zero_n, cudaStream_t stream);

// dQ: one (query tile, q-head) item per CTA, same key walk as the forward.
// When `dq_prompt` is not null, prompt rows are also written there in fp32
// ([prompt rows of all groups in accumulator order, Hq, d]).
cudaError_t launch_dq(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK,
                      const CUtensorMap& mV, const CUtensorMap& mdO, const float* lse, const float* Dvec,
                      void* dq, float* dq_prompt, unsigned int* err, cudaStream_t stream);

// dK/dV: one (key tile, kv-head, split) item per CTA.  Response key rows are
// written to dk/dv (bf16); prompt key rows go to fp32 `acc_k/acc_v`
// ([P,Hkv,d]) with atomics when `deterministic` is 0, or to the split's slice
// of `part_k/part_v` ([S,P,Hkv,d]) when it is 1.  With `dq_acc` not null
// (atomic mode only) the kernel also adds every tile's dQ (unscaled) to the
// fp32 accumulator dq_acc [Hq][d/4][T][4], which must start at zero.
cudaError_t launch_dkdv(const Sched& s, int d, const CUtensorMap& mQ, const CUtensorMap& mK,
                        const CUtensorMap& mV, const CUtensorMap& mdO, const float* lse, const float* Dvec,
                        void* dk, void* dv, float* acc_k, float* acc_v, float* dq_acc, int deterministic,
                        unsigned int* err, cudaStream_t stream);

// dq [T,Hq,d] bf16 = scale * dq_acc ([Hq][d/4][T][4] fp32), RNE.  Rows t <
// prompt_end outside [keep_lo, keep_hi) are left untouched; when dq_prompt
// is not null, rows t < prompt_end inside it are also written there in fp32
// ([prompt_end, Hq, d]).
cudaError_t launch_dq_cast(const float* dq_acc, void* dq, float* dq_prompt, int64_t T, int Hq, int d, float scale,
                           int64_t prompt_end, int64_t keep_lo, int64_t keep_hi, cudaStream_t stream);

// Where each group's prompt rows sit: accumulator rows [acc_row[g],
// acc_row[g+1]) hold the prompt that starts at packed row packed_row[g].
struct PromptMap {
  int32_t ngroups;
  int32_t acc_row[kMaxSeg + 1];
  int32_t packed_row[kMaxSeg];
};

// Prompt rows of dK/dV: sum the `nsplit` fp32 slices (stride `slice` floats)
// of the accumulator in split order and round to bf16 (RNE) into the
// prompt rows of dk/dv (row_elems = Hkv * d values per row).  When f32_k /
// f32_v are not null, the fp32 sums are also stored there, in accumulator
// row order ([prompt rows of all groups, Hkv, d]).
cudaError_t launch_prompt_reduce(const float* src_k, const float* src_v, int nsplit, size_t slice,
                                 void* dk, void* dv, float* f32_k, float* f32_v, const PromptMap& map,
                                 int row_elems, unsigned int* err, cudaStream_t stream);

// Device address of the library's error word on the current device (looked
// up once per device), or null.
unsigned int* device_error_word();

// Records the CUDA code behind a failure (a cudaError_t, or the driver result
// of a rejected tensor map) for the calling thread's dualkv_last_cuda_error
// and returns DUALKV_ERR_CUDA.
int cuda_fail(int code);
inline int cuda_fail(cudaError_t e) { return cuda_fail(static_cast<int>(e)); }
int last_cuda_error();

// Self-test of the bounded waits: a wait on an mbarrier phase that never
// completes gives up after limit_ns and records a timeout at `site`.
cudaError_t launch_wait_timeout_selftest(unsigned int* err, uint64_t limit_ns, uint32_t site, cudaStream_t stream);

}  // namespace dkv
