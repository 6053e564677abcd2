// mha_wait.cuh - the bounded mbarrier waits every kernel of the library
// uses, and the bits they record in the per-device status word.
//
// A wait that runs past its cycle budget sets a timeout bit plus a bit naming
// the wait site in the status word, raises the CTA's abort flag (which ends
// every other wait of that CTA at once) and returns false; the caller then
// leaves its loop, drains its own copies and MMAs, and exits normally.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace mha {

// Bits of the device status word.
constexpr unsigned kStatusTimeout = 1u << 31;
enum WaitSite : unsigned {
  kSiteProducerEmpty = 1u << 0,
  kSiteMmaQ = 1u << 1,
  kSiteMmaKV = 1u << 2,
  kSiteMmaP = 1u << 3,
  kSiteSoftmaxS = 1u << 4,
  kSiteSoftmaxO = 1u << 5,
  kSiteDrain = 1u << 6,
  kSiteSelftest = 1u << 7,
};

struct WaitCtl {
  volatile int* abort;
  unsigned* status;
  long long limit;
};

__device__ __forceinline__ void raise_timeout(const WaitCtl& c, unsigned site) {
  *c.abort = 1;
  atomicOr(c.status, kStatusTimeout | site);
}

// Bounded wait by a single thread.  Returns false on abort or timeout.
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                         unsigned site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*c.abort) return false;
    if (clock64() - t0 > c.limit) {
      raise_timeout(c, site);
      return false;
    }
  }
  return true;
}

// Bounded wait by a whole warp, with a warp-uniform outcome (the warp goes
// on to execute .sync.aligned tcgen05 instructions together).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                          unsigned site) {
  // the clock is read only once the first probe has failed: on the fast
  // path (barrier already complete) it would be most of the cost
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    const uint32_t ok = ptx::mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*c.abort)
        stop = 1;
      else if (clock64() - t0 > c.limit)
        stop = 2;
    }
    stop = __shfl_sync(0xffffffffu, stop, 0);
    if (stop) {
      if (stop == 2 && (threadIdx.x & 31) == 0) raise_timeout(c, site);
      return false;
    }
  }
}

// Wait with its own budget that ignores the abort flag: used only to drain
// copies / MMAs this CTA started before it frees its resources.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > c.limit) {
      atomicOr(c.status, kStatusTimeout | kSiteDrain);
      return;
    }
  }
}

}  // namespace mha
