// fa_device_common.cuh — bounded barrier waits shared by the forward kernels.
//
// Every wait on an mbarrier spins for at most `limit` clock64 cycles. When it
// gives up it records a timeout (and where) in the device status word, raises
// the CTA's abort flag so that the other roles stop waiting too, and returns
// false; the caller then drains its own asynchronous work, frees tensor memory
// and exits. Nothing traps.
#pragma once

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

struct WaitCtl {
  volatile int* abort_flag;  // shared memory, one per CTA
  unsigned int* status;      // [0] flags, [1] where
  long long limit;
};

__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const WaitCtl& ctl, unsigned where,
                                           bool honour_abort) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *ctl.abort_flag) return false;
    if (clock64() - t0 > ctl.limit) {
      atomicOr(ctl.status, kStatusTimeout);
      atomicCAS(ctl.status + 1, 0u, where);
      *ctl.abort_flag = 1;
      return false;
    }
  }
}

// Wait for the phase of parity `parity` of `bar` to complete.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& ctl, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, ctl, where, true);
}

// Whole-warp wait with a warp-uniform outcome.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const WaitCtl& ctl, unsigned where) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ctl, where));
}

// Same, but keeps waiting after another role aborted (used to drain in-flight copies/MMAs).
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, ctl, kWhereDrain, false);
}

// Testing build only: clock64 stamp of pipeline event `ev` for tile `j`.
#ifdef FA_TESTING
#define FA_TRACE(p, ev, j)                                                                                 \
  do {                                                                                                     \
    if ((p).timeline && blockIdx.x < kTraceCtas && (j) < kTraceTiles)                                     \
      (p).timeline[(static_cast<size_t>(blockIdx.x) * kTraceEvents + (ev)) * kTraceTiles + (j)] = clock64(); \
  } while (0)
#else
#define FA_TRACE(p, ev, j) \
  do {                     \
  } while (0)
#endif

}  // namespace fa
