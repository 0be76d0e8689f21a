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

// Everything a bounded wait needs: the CTA's abort flag (a shared-memory
// address) and the kernel parameters (status word, wait limit). Kept small:
// once inlined, the parameter reads come from the kernel's parameter space.
// P is the kernel's parameter block (FwdParams or BwdParams).
template <class P>
struct WaitCtlT {
  const P& p;           // the kernel's __grid_constant__ parameters
  uint32_t abort_addr;  // shared-memory address of the CTA's abort flag
};
using WaitCtl = WaitCtlT<FwdParams>;

__device__ __forceinline__ int abort_raised(uint32_t addr) {
  int v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <class P>
static __device__ __forceinline__ void record_timeout(const P& p, uint32_t abort_addr, unsigned where) {
  atomicOr(p.status, kStatusTimeout);
  atomicCAS(p.status + 1, 0u, where);
  asm volatile("st.volatile.shared.s32 [%0], %1;" ::"r"(abort_addr), "r"(1) : "memory");
}

template <class Ctl>
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const Ctl& ctl, unsigned where,
                                              bool honour_abort) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && abort_raised(ctl.abort_addr)) return false;
    if (clock64() - t0 > ctl.p.wait_limit) {
      record_timeout(ctl.p, ctl.abort_addr, where);
      return false;
    }
  }
}

// Wait for the phase of parity `parity` of `bar` to complete.
template <class Ctl>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& ctl, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, ctl, where, true);
}

// Whole-warp wait with a warp-uniform outcome.
template <class Ctl>
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Ctl& ctl, unsigned where) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ctl, where));
}

// Same, but keeps waiting after another role aborted (used to drain in-flight copies/MMAs).
template <class Ctl>
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, ctl, kWhereDrain, false);
}

// The lazy-rescale threshold in log2 units: the reference max of a row moves
// only when P taken against it would exceed 2^threshold (the kernels test
// each tile's max against it), so P <= 2^threshold (fits fp16 and bf16). The
// testing build takes it
// from the parameters, so that 0 (rescale whenever the max grows, the
// dataflow page's section 2.3) can be run against the oracle too.
__device__ __forceinline__ float rescale_threshold(const FwdParams& p) {
#ifdef FA_TESTING
  return p.rescale_tau;
#else
  (void)p;
  return kRescaleThresholdLog2;
#endif
}

// Host side: launch `kern` as a programmatic dependent of the previous kernel
// in `stream` (it may start while that kernel's last CTAs still run; it
// must itself wait, griddepcontrol.wait, before it reads that kernel's
// results or, reading none, before it completes).
template <class Kern, class... Args>
inline cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
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
