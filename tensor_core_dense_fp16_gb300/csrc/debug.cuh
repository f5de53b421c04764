// debug.cuh — device-side checks of the -DHGEMM_DEBUG build.
//
// Every shared-memory address a PTX wrapper (ptx.cuh) hands to a barrier,
// a TMA copy, an asynchronous copy, a bulk copy or ldmatrix is checked to lie
// inside the CTA's own shared memory, every TMA copy's innermost coordinate
// to be 16-byte aligned (8 FP16 elements), every TMEM load to stay inside the
// 512 columns, and the kernels that address global memory themselves (the
// generic, substitution and elementwise kernels, the fused epilogue's reads
// of C and the bias) check each computed index against the extent it must
// stay in. A failed check records a code in its translation unit's debug
// word and SKIPS the access (a copy that is skipped leaves its barrier
// short, so the waiting side runs into its bounded wait and the kernel
// leaves with the watchdog code set): no trap, no fault. The host reads and
// clears the words in hgemm_device_status, which then returns
// HGEMM_ERR_DEBUG_CHECK; hgemm_debug_code tells which check fired.
//
// Without HGEMM_DEBUG every check compiles to nothing. The predicates are
// plain host/device functions so that the host-side self test
// (hgemm_debug_selftest) exercises the same code on values outside the
// ranges, which no GPU run may do.
#pragma once

#include <cstdint>

#include <cstdio>

#include <cuda_runtime.h>

namespace hg {

// Codes recorded by a failed check (distinct from the watchdog codes).
enum DebugCode : int {
  kDbgSmemRange = 101,    // a shared-memory access outside the CTA's shared memory
  kDbgTmaCoord = 102,     // a TMA innermost coordinate not 16-byte aligned
  kDbgTmemRange = 103,    // a TMEM access past lane 127 or column 511
  kDbgGlobalIndex = 104,  // a computed global index outside its extent
  kDbgAlign = 105,        // a vector access not aligned to its width
};

// [addr, addr + bytes) inside [lo, lo + size).
__host__ __device__ constexpr bool dbg_range_ok(uint32_t addr, uint32_t bytes, uint32_t lo, uint32_t size) {
  return addr >= lo && bytes <= size && addr - lo <= size - bytes;
}

// A TMA innermost coordinate of elements of `elem_bytes` bytes.
__host__ __device__ constexpr bool dbg_tma_x_ok(int32_t x, int32_t elem_bytes) {
  return (static_cast<int64_t>(x) * elem_bytes) % 16 == 0;
}

// A TMEM address (lane << 16 | column) read `cols` columns wide.
__host__ __device__ constexpr bool dbg_tmem_ok(uint32_t taddr, uint32_t cols) {
  return (taddr >> 16) < 128u && (taddr & 0xFFFFu) + cols <= 512u;
}

// 0 <= i < n.
__host__ __device__ constexpr bool dbg_index_ok(int64_t i, int64_t n) { return i >= 0 && i < n; }

// An address aligned to `bytes`.
__host__ __device__ constexpr bool dbg_aligned(uint64_t addr, uint64_t bytes) { return addr % bytes == 0; }

#if defined(HGEMM_DEBUG) && defined(__CUDACC__)
namespace {
__device__ int g_debug_word = 0;  // one per translation unit
}  // namespace

__device__ __forceinline__ bool dbg_report(bool ok, int code) {
  if (!ok) atomicCAS(&g_debug_word, 0, code);
  return ok;
}

// The CTA's own shared memory. In its window the reserved region (its
// capacity, 1 KB on this GPU) comes first, then the static and the dynamic
// shared memory, which %total_smem_size counts (measured: dynamic shared
// memory starts at the capacity when there is no static shared memory).
// Inside a cluster a CTA's own addresses carry its window in the bits above
// the low 24 (rank 1's start at 1 << 24; measured), so the window is taken
// from the CTA's own dynamic shared memory, and an address in another
// window fails the check.
__device__ __forceinline__ bool dbg_smem(uint32_t addr, uint32_t bytes) {
  extern __shared__ __align__(16) uint8_t hg_dbg_dynamic_smem[];
  const uint32_t window = static_cast<uint32_t>(__cvta_generic_to_shared(hg_dbg_dynamic_smem)) & 0xFF000000u;
  uint32_t cap, size;
  asm volatile("mov.u32 %0, %%reserved_smem_offset_cap;" : "=r"(cap));
  asm volatile("mov.u32 %0, %%total_smem_size;" : "=r"(size));
  const uint32_t lo = window + cap;
  const bool ok = dbg_range_ok(addr, bytes, lo, size);
  if (!ok && atomicCAS(&g_debug_word, 0, kDbgSmemRange) == 0)
    printf("hgemm debug check: shared-memory access [%u, +%u) outside [%u, +%u), block %d thread %d\n", addr,
           bytes, lo, size, static_cast<int>(blockIdx.x), static_cast<int>(threadIdx.x));
  return ok;
}

#define HG_DBG_SMEM(addr, bytes) (::hg::dbg_smem((addr), (bytes)))
#define HG_DBG_TMA_X(x) (::hg::dbg_report(::hg::dbg_tma_x_ok((x), 2), ::hg::kDbgTmaCoord))
#define HG_DBG_TMEM(taddr, cols) (::hg::dbg_report(::hg::dbg_tmem_ok((taddr), (cols)), ::hg::kDbgTmemRange))
#define HG_DBG_INDEX(i, n) (::hg::dbg_report(::hg::dbg_index_ok((i), (n)), ::hg::kDbgGlobalIndex))
#define HG_DBG_ALIGN(p, bytes) \
  (::hg::dbg_report(::hg::dbg_aligned(reinterpret_cast<uint64_t>(p), (bytes)), ::hg::kDbgAlign))
// Host accessor of this translation unit's word (see HG_DEBUG_WORD_ACCESSOR).
#define HG_DEBUG_WORD_ACCESSOR(name)                                       \
  cudaError_t debug_word_##name(int** out) {                               \
    return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_debug_word); \
  }
#else
#define HG_DBG_SMEM(addr, bytes) (true)
#define HG_DBG_TMA_X(x) (true)
#define HG_DBG_TMEM(taddr, cols) (true)
#define HG_DBG_INDEX(i, n) (true)
#define HG_DBG_ALIGN(p, bytes) (true)
#define HG_DEBUG_WORD_ACCESSOR(name)         \
  cudaError_t debug_word_##name(int** out) { \
    *out = nullptr;                          \
    return cudaSuccess;                      \
  }
#endif

}  // namespace hg
