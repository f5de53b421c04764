// kernel_common.cuh — device helpers shared by the tensor-core kernels:
// tile rasterisation, the bounded-wait watchdog and FP16 packing.
#pragma once

#include <cuda_fp16.h>

#include "debug.cuh"
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

// ------------------------------------------------------- fused epilogue

// One output of the fused epilogue, in FP32: alpha·acc + beta·c_old +
// bias, then the ReLU (a NaN stays NaN). `c_old` is used in mode 2 only and
// `b` is the column's bias (0 without one).
__device__ __forceinline__ float epi_value(float acc, const EpiArgs& e, float c_old, float b) {
  float x = e.alpha * acc;
  if (e.mode == 2) x = fmaf(e.beta, c_old, x);
  x += b;
  if (e.relu && x < 0.f) x = 0.f;
  return x;
}

// The previous FP16 values C[row, col0 .. col0+7] (mode 2), zeros outside C.
// col0, N and the row pitch ldc are multiples of 8 (TMA paths), so each
// read is one aligned 16-byte load inside row `row`.
__device__ __forceinline__ uint4 load_c_old8(const EpiArgs& e, const uint16_t* C, int64_t M,
                                             int64_t N, int64_t ldc, int64_t row, int64_t col0) {
  if (e.mode != 2 || row >= M || col0 >= N) return make_uint4(0u, 0u, 0u, 0u);
  const uint16_t* src = C + row * ldc + col0;
  if (!HG_DBG_INDEX(col0 + 7, N) || !HG_DBG_ALIGN(src, 16)) return make_uint4(0u, 0u, 0u, 0u);
  return *reinterpret_cast<const uint4*>(src);
}

// Mode 2: asks L2 for the previous C values of row `grow`, columns
// [x0, x0 + ncols), while the tile's MMAs still run (one request per 64
// bytes, so rows that straddle 128-byte lines are covered).
__device__ __forceinline__ void prefetch_c_row(const EpiArgs& e, const uint16_t* C, int64_t M,
                                               int64_t N, int64_t ldc, int64_t grow, int64_t x0,
                                               int ncols) {
  if (e.mode != 2 || grow >= M) return;
  for (int c = 0; c < ncols; c += 32)
    if (x0 + c < N) asm volatile("prefetch.global.L2 [%0];" ::"l"(C + grow * ldc + x0 + c));
}

// The biases of columns col0 .. col0+7 (zeros past N or without a bias);
// col0 is a multiple of 8, so with a 16-byte-aligned bias one vector load.
__device__ __forceinline__ uint4 load_bias8(const EpiArgs& e, int64_t col0, int64_t N) {
  if (!e.bias || col0 >= N) return make_uint4(0u, 0u, 0u, 0u);
  if ((reinterpret_cast<uintptr_t>(e.bias) & 15u) == 0 && col0 + 8 <= N)
    return __ldg(reinterpret_cast<const uint4*>(e.bias + col0));
  uint16_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = col0 + i < N ? __ldg(e.bias + col0 + i) : static_cast<uint16_t>(0);
  return make_uint4(h[0] | (static_cast<uint32_t>(h[1]) << 16), h[2] | (static_cast<uint32_t>(h[3]) << 16),
                    h[4] | (static_cast<uint32_t>(h[5]) << 16), h[6] | (static_cast<uint32_t>(h[7]) << 16));
}

// Eight accumulators (FP32 bits) through the fused epilogue with their
// previous values and biases, packed to FP16 (round to nearest even).
__device__ __forceinline__ uint4 epi_pack8(const uint32_t* v, const EpiArgs& e, uint4 c_old,
                                           uint4 bias8) {
  const __half* ch = reinterpret_cast<const __half*>(&c_old);
  const __half* bh = reinterpret_cast<const __half*>(&bias8);
  float f[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    f[i] = epi_value(__uint_as_float(v[i]), e, __half2float(ch[i]), __half2float(bh[i]));
  uint4 r;
  r.x = pack_half2(__float_as_uint(f[0]), __float_as_uint(f[1]));
  r.y = pack_half2(__float_as_uint(f[2]), __float_as_uint(f[3]));
  r.z = pack_half2(__float_as_uint(f[4]), __float_as_uint(f[5]));
  r.w = pack_half2(__float_as_uint(f[6]), __float_as_uint(f[7]));
  return r;
}

}  // namespace hg

namespace hg {

// Row `lane` of a staged 32×64 box of C: the 64 accumulators of that row
// (v0: columns x0 .. x0+31, v1: x0+32 .. x0+63) rounded to FP16 (through the
// fused epilogue when FUSED) into the 128-byte-swizzled staging row `row`
// (16-byte chunk j at position j ^ (lane % 8)). grow: the row of C.
template <bool FUSED>
__device__ __forceinline__ void stage_row64(uint8_t* row, int lane, const uint32_t (&v0)[32],
                                            const uint32_t (&v1)[32], const EpiArgs& e,
                                            const uint16_t* C, int64_t M, int64_t N, int64_t ldc,
                                            int64_t grow, int64_t x0) {
  if constexpr (!FUSED) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t* v = (j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4));
      uint4 pk;
      pk.x = pack_half2(v[0], v[1]);
      pk.y = pack_half2(v[2], v[3]);
      pk.z = pack_half2(v[4], v[5]);
      pk.w = pack_half2(v[6], v[7]);
      *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = pk;
    }
    return;
  }
  uint4 c_old[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) c_old[j] = load_c_old8(e, C, M, N, ldc, grow, x0 + 8 * j);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t* v = (j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4));
    *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) =
        epi_pack8(v, e, c_old[j], load_bias8(e, x0 + 8 * j, N));
  }
}

}  // namespace hg
