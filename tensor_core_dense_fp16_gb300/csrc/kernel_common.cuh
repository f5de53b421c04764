// kernel_common.cuh — device helpers shared by the tensor-core kernels:
// tile rasterisation, the bounded-wait watchdog and FP16 packing.
#pragma once

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace hg {

// Grouped raster: tiles are numbered so that GROUP_M consecutive M-tiles
// share each N-tile before moving to the next N-tile.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
  const int per_group = group_m * num_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
  // odd groups walk N backwards, so a group starts on the B columns the
  // previous group used last (still in L2)
  if (g & 1) nb = num_n - 1 - nb;
}

struct Watchdog {
  volatile int* abort_flag;  // shared memory, CTA-wide
  int* status;               // global watchdog word
  unsigned long long timeout_ns;

  __device__ void raise(int code) const {
    *abort_flag = 1;
    atomicCAS(status, 0, code);
  }
};

// Waits for phase `parity` of `bar`. Returns false if another role raised the
// abort flag or if `timeout_ns` passed (then this wait raises it itself).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                           int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*wd.abort_flag) return false;
    if (globaltimer_ns() - t0 > wd.timeout_ns) {
      wd.raise(code);
      return false;
    }
  }
  return true;
}

// The same with cluster-scope acquire, for barriers that other threads of
// the cluster arrive on remotely (ordinary arrivals carry their release to
// the waiter only at cluster scope). Barriers completed by TMA transaction
// bytes or by tcgen05.commit, even from the other CTA of a pair, are waited
// on at CTA scope.
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity,
                                                   const Watchdog& wd, int code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (*wd.abort_flag) return false;
    if (globaltimer_ns() - t0 > wd.timeout_ns) {
      wd.raise(code);
      return false;
    }
  }
  return true;
}

// Drain wait: ignores the abort flag (the copy or MMA must land before the
// CTA's memory goes away) but is still bounded.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const Watchdog& wd) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > wd.timeout_ns) {
      wd.raise(kWdDrain);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool wait_drain_cluster(uint32_t bar, uint32_t parity,
                                                   const Watchdog& wd) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > wd.timeout_ns) {
      wd.raise(kWdDrain);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace hg
