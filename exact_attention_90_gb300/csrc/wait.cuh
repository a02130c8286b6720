// wait.cuh -- bounded mbarrier waits.
//
// No wait in these kernels spins forever.  A wait that has not completed after
// FA_WAIT_BUDGET_CYCLES SM clocks (about a second) records an error bit in a
// device word, raises the CTA's abort flag and returns false; once the flag is
// up every later wait of the CTA returns at once, so all roles run through
// their (now meaningless) loops, free tensor memory and exit.  The host reads
// the word with fa_debug_sync_check().  drain() is the final, also bounded,
// wait for a CTA's own copies or MMAs still in flight; it ignores the flag.
#pragma once

#include <cstdint>

#include "ptx.cuh"

#ifndef FA_WAIT_BUDGET_CYCLES
#define FA_WAIT_BUDGET_CYCLES (1ll << 31)
#endif

namespace fa {

// error bits (which role gave up)
enum : unsigned int {
  kErrWaitLoad = 1u << 0,
  kErrWaitMma = 1u << 1,
  kErrWaitSoftmax = 1u << 2,
  kErrWaitEpilogue = 1u << 3,
  kErrDrain = 1u << 4,
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err, unsigned int code,
                                         long long budget = FA_WAIT_BUDGET_CYCLES) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      atomicOr(err, code);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool drain_bar(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > FA_WAIT_BUDGET_CYCLES) {
      atomicOr(err, kErrDrain);
      return false;
    }
  }
  return true;
}

}  // namespace fa
