// Device-side checks of the checks build (compiled with -DDUALKV_CHECKS).
//
// The checks stand where a memory sanitizer cannot run: before each global
// access and each tensor-copy coordinate the kernels compute, `check` tests
// the index against the extent it must stay inside; at the end of a CTA every
// pipeline role compares the number of steps it completed with the number
// the schedule gave it.  A failed check never traps: it records
// kDevErrCheck and the site in the device error word (first error wins) and
// returns false, and the caller skips the access.  In the regular build
// `check` is the constant true and compiles away.
#pragma once

#include "ptx.cuh"

namespace dkv {

enum : uint32_t { kDevErrCheck = 7u };

#ifdef DUALKV_CHECKS
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif

__device__ __forceinline__ bool check(bool cond, unsigned int* err, uint32_t site) {
  if (!kChecks || cond) return true;
  record_error(err, kDevErrCheck, site);
  return false;
}

// Index i inside [0, n).
__device__ __forceinline__ bool check_index(int64_t i, int64_t n, unsigned int* err, uint32_t site) {
  return check(i >= 0 && i < n, err, site);
}

// Per-CTA step counters of the pipeline roles (shared memory, checks build):
// each role stores its completed steps, and after the CTA's final barrier one
// thread compares them with the expected count.
struct RoleSteps {
  int32_t* slot;  // kRoles ints in shared memory (producer, MMA issuer, two consumer groups)
  static constexpr int kRoles = 4;

  __device__ __forceinline__ void init() const {
    if constexpr (kChecks) {
      for (int r = 0; r < kRoles; ++r) slot[r] = -1;
    }
  }
  __device__ __forceinline__ void put(int role, int32_t steps) const {
    if constexpr (kChecks) slot[role] = steps;
  }
  // Every role that reported must have completed `expected` steps.  A role
  // that stopped early on a timed-out wait has already recorded that error,
  // which this one does not replace.
  __device__ __forceinline__ void verify(int32_t expected, unsigned int* err, uint32_t site) const {
    if constexpr (kChecks) {
      for (int r = 0; r < kRoles; ++r)
        if (slot[r] != -1) check(slot[r] == expected, err, site);
    }
  }
};

}  // namespace dkv
