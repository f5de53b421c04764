// hgemm_trsm_chain.cu — the triangular solve with a workspace, after the
// inverses of its diagonal blocks are known, as ONE persistent launch.
//
// What it computes: the solve of "异构计算中高性能TRMM与TRSM的递归算法实现"
// (§2.1–2.3; Aᵀ·X = alpha·B, or the page's literal A·X = alpha·B), with the
// diagonal blocks of order ≤ 512 applied through their inverses (FP16, in
// the workspace). Unrolled over those blocks, in the order the recursion
// solves them, the solve is a chain of products on Xᵀ (m × n, row-major with
// pitch ldx: column j of X is row j of Xᵀ):
//   product of block b   Xᵀ_b := Xᵀ_b · L_b⁻¹     (A·X = B: · L_b⁻ᵀ)
//   update after block b Xᵀ_c −= Xᵀ_b · A(b, c)   for every block c not yet
//                        solved (A·X = B: · A(c, b)ᵀ), as one product over
//                        all their columns,
// each phase reading what the one before wrote. The recursion sums the same
// terms; here each block's contribution is subtracted (and X rounded to
// FP16) as soon as that block is solved, so that every phase but the
// products spreads over all remaining columns (right-looking order).
//
// How (a chain of latency-bound launches turned into one):
//   * a cooperative launch of one CTA per SM (all CTAs co-resident); phases
//     are separated by a grid-wide barrier: an arrival counter in the
//     workspace (released at GPU scope, polled with acquire, bounded in time);
//   * phase 0 (unless the solve is in place with alpha = 1): X := alpha·B,
//     grid-stride, FP32 product rounded to FP16;
//   * every other phase is a set of bm × bn output tiles (bm 64 or 128, bn
//     64, 128 or 256, chosen per phase by the host so that the tiles fill the
//     grid with the fewest operand bytes per SM), one or more per CTA, each
//     a K ≤ 512 tcgen05 product: warp 0 streams 64 × 64 TMA boxes of Xᵀ and
//     of the second operand (an inverse, or the triangle itself, K- or
//     N-contiguous) into a ring of 128-byte-swizzled stages whose geometry
//     follows the phase's tile; warp 1 issues the M=128 MMAs into one of two
//     256-column FP32 accumulators in TMEM (a 64-row tile leaves half of them
//     unused); warps 2–5 read the accumulator with tcgen05.ld, subtract it
//     from the previous X (updates) or take it as it is (products), round to
//     FP16 and store with plain 16-byte stores;
//   * the second operand never changes during the launch, so the producer
//     loads the next phase's first stages of it before the barrier, and only
//     the Xᵀ boxes wait for it;
//   * a product overwrites the columns it reads, and the tiles of one row
//     range read each other's columns: each 64-row group of Xᵀ has a counter
//     that the MMA issuer of every tile covering it raises once the tile's
//     Xᵀ boxes have landed; the epilogue stores only when the counter has
//     reached the phase's target (all of a product phase's tiles run at
//     once: the host keeps them within the grid);
//   * writes of one phase reach the next through the barrier: every thread's
//     stores, a CTA barrier, a GPU-scope release by one thread; on the other
//     side an acquire, a proxy fence (TMA reads come next) and a CTA barrier.
//     Reads of X by the epilogue bypass L1 (ld.global.cg).
//   * Every wait is bounded. A wait that gives up records a watchdog code,
//     raises the CTA's abort flag and, at the next barrier, the launch's
//     abort word, which every CTA polls; all then drain their copies and
//     MMAs, free TMEM and return.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

constexpr int kThreads = 192;                     // producer, MMA issuer, four epilogue warps
constexpr int kRingBytes = 192 * 1024;            // operand ring, regrouped into stages per phase
constexpr int kMaxStages = 8;
constexpr int kASlot = kTcBM * kTcBK * 2;         // 16 KB: an M=128 MMA reads 128 rows of Xᵀ
constexpr int kBox = 64;                          // every TMA box is 64 × 64 elements
constexpr int kBoxBytes = kBox * kBox * 2;        // 8 KB
constexpr int kAccCols = 256;                     // the widest tile: 256 FP32 columns
constexpr int kTmemCols = 2 * kAccCols;           // two accumulators
constexpr int kOffBar = kRingBytes;
// full, empty, accumulator full ×2 / empty ×2, drain
constexpr int kNumBars = 2 * kMaxStages + 4 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM address, abort flag, barriers passed, epilogue verdict
constexpr int kOffPhases = kOffMisc + 16;         // the phase table, copied from the parameters
constexpr int kSmemBytes = kOffPhases + kChainMaxPhases * static_cast<int>(sizeof(ChainPhase)) + 1024;
constexpr int kEpiThreads = 128;                  // warps 2–5
constexpr int kEpiBarrier = 1;                    // named barrier of the epilogue warps
static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(kRingBytes / (kASlot + 64 * kTcBK * 2) >= kMaxStages, "the narrowest stages fill the ring");

// A phase, decoded.
struct Phase {
  int kind, b_map, b_mn, bm, bn;
  int num_m, num_n, num_tiles;
  int n0, n_end, k0, ksteps, b_kbase, b_nbase;
  uint32_t rg_target;
  int stages;
  uint32_t stage_bytes, tx_bytes;
};

__device__ __forceinline__ Phase decode(const ChainPhase& c, int m) {
  Phase p;
  p.kind = c.flags & 3;
  p.b_map = (c.flags >> 2) & 3;
  p.b_mn = (c.flags >> 4) & 1;
  p.bm = ((c.flags >> 5) & 3) * 64;
  p.bn = ((c.flags >> 8) & 7) * 64;
  p.n0 = c.n0;
  p.n_end = c.n_end;
  p.k0 = c.k0;
  p.ksteps = c.ksteps;
  p.b_kbase = c.b_kbase;
  p.b_nbase = c.b_nbase;
  p.rg_target = c.rg_target;
  if (p.kind == kChainCopy || p.bm == 0 || p.bn == 0) {
    p.num_m = p.num_n = p.num_tiles = 0;
    p.stages = 1;
    p.stage_bytes = p.tx_bytes = 0;
    return p;
  }
  p.num_m = (m + p.bm - 1) / p.bm;
  p.num_n = (p.n_end - p.n0 + p.bn - 1) / p.bn;
  p.num_tiles = p.num_m * p.num_n;
  p.stage_bytes = static_cast<uint32_t>(kASlot + p.bn * kTcBK * 2);
  p.stages = min(kMaxStages, static_cast<int>(kRingBytes / p.stage_bytes));
  p.tx_bytes = static_cast<uint32_t>((p.bm / kBox + p.bn / kBox) * kBoxBytes);
  return p;
}

// Tile t of a phase: row tile mi, column tile ni (column-tile major, so that
// concurrently running tiles share the second operand's boxes).
__device__ __forceinline__ void tile_of(const Phase& ph, int t, int& mi, int& ni) {
  ni = t / ph.num_m;
  mi = t - ni * ph.num_m;
}

__device__ __forceinline__ const CUtensorMap* map_b(const Phase& ph, const CUtensorMap* w,
                                                    const CUtensorMap* wr, const CUtensorMap* a) {
  return ph.b_map == kChainMapW ? w : ph.b_map == kChainMapWRagged ? wr : a;
}

// The second operand's boxes of k-step kk of column tile ni into `sb`.
__device__ __forceinline__ void load_b(const Phase& ph, const CUtensorMap* map, uint32_t sb, uint32_t bar,
                                       int ni, int kk) {
  const int kc = ph.b_kbase + kk * kTcBK;
  for (int i = 0; i < ph.bn / kBox; ++i) {
    const int nc = ph.b_nbase + ni * ph.bn + i * kBox;
    if (ph.b_mn)
      tma_load_2d(sb + i * kBoxBytes, map, bar, nc, kc);  // box: 64 N (contiguous) × 64 K rows
    else
      tma_load_2d(sb + i * kBoxBytes, map, bar, kc, nc);  // box: 64 N rows × 64 K (contiguous)
  }
}

// The Xᵀ boxes of k-step kk of row tile mi into `sa`.
__device__ __forceinline__ void load_a(const Phase& ph, const CUtensorMap* map, uint32_t sa, uint32_t bar,
                                       int mi, int kk) {
  for (int i = 0; i < ph.bm / kBox; ++i)
    tma_load_2d(sa + i * kBoxBytes, map, bar, ph.k0 + kk * kTcBK, mi * ph.bm + i * kBox);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The launch's abort word: set by a CTA that gave up, polled by every wait
// on other CTAs.
__device__ __forceinline__ bool launch_aborted(const ChainArgs& p) {
  return ld_relaxed_gpu(p.sync + kChainSyncAbort) != 0u;
}

__device__ __forceinline__ void st_release_cta(volatile uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(const_cast<uint32_t*>(p))), "r"(v)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta(const volatile uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];"
               : "=r"(v)
               : "r"(smem_u32(const_cast<const uint32_t*>(p)))
               : "memory");
  return v;
}

// Grid-wide barrier number `index` (1, 2, ...), by the epilogue warps, the
// only ones that write X: their stores, a named barrier, then one thread
// releases the CTA's arrival at GPU scope and polls the count with acquire;
// it publishes the outcome (`epi_ok`, read by every epilogue thread after
// the second named barrier, so all four warps decide alike) and, on
// success, the number of barriers passed (`passed`, released at CTA scope
// for the producer, which fences its own TMA reads behind it). Returns false
// when the launch is aborting (this CTA's abort flag, the launch's abort
// word, or the bounded wait gave up).
__device__ bool grid_barrier(const ChainArgs& p, uint32_t index, volatile int* abort_flag,
                             volatile uint32_t* passed, volatile int* epi_ok) {
  named_bar_sync(kEpiBarrier, kEpiThreads);  // every epilogue store of the phase precedes the release
  if (threadIdx.x == 64) {
    uint32_t* ctr = p.sync + kChainSyncBarrier;
    bool ok = *abort_flag == 0;
    if (!ok) atomicExch(p.sync + kChainSyncAbort, 1u);
    red_release_gpu(ctr, 1u);
    const uint32_t target = index * gridDim.x;
    if (ok && ld_acquire_gpu(ctr) < target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(ctr) < target) {
        if (*abort_flag || launch_aborted(p)) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          atomicCAS(p.status, 0, kWdGridBarrier);
          atomicExch(p.sync + kChainSyncAbort, 1u);
          ok = false;
          break;
        }
      }
    }
    if (!ok) *abort_flag = 1;
    *epi_ok = ok ? 1 : 0;
    if (ok) st_release_cta(passed, index);
  }
  named_bar_sync(kEpiBarrier, kEpiThreads);
  return *epi_ok != 0;
}

// The producer's wait for grid barrier `index` (the epilogue's leader
// publishes it); false when the CTA is aborting or the bounded wait gave up.
__device__ bool wait_passed(const volatile uint32_t* passed, uint32_t index, const Watchdog& wd) {
  if (ld_acquire_cta(passed) >= index) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_cta(passed) < index) {
    if (*wd.abort_flag) return false;
    if (globaltimer_ns() - t0 > wd.timeout_ns) {
      wd.raise(kWdGridBarrier);
      return false;
    }
  }
  return true;
}

// Phase 0: X := alpha·B over the n × m column-major operands, by the
// epilogue warps (every element read and written by the same thread, so
// X == B works); four loads in flight per thread.
__device__ void copy_phase(const ChainArgs& p) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kEpiThreads + (threadIdx.x - 64);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kEpiThreads;
  constexpr int U = 4;
  if (p.copy_vec) {
    const int64_t per = p.n / 8, count = per * p.m;
    for (int64_t t0 = tid; t0 < count; t0 += U * stride) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + u * stride;
        if (t < count) {
          const int64_t j = t / per, i = (t - j * per) * 8;
          const uint16_t* src = p.B + j * p.ldb + i;
          v[u] = HG_DBG_ALIGN(src, 16) ? __ldcg(reinterpret_cast<const uint4*>(src)) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + u * stride;
        if (t >= count) break;
        const int64_t j = t / per, i = (t - j * per) * 8;
        uint16_t* dst = p.X + j * p.ldx + i;
        if (!HG_DBG_ALIGN(dst, 16)) continue;
        uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
          const __half2 h = __floats2half2_rn(p.alpha * f.x, p.alpha * f.y);
          w[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
    const int64_t count = static_cast<int64_t>(p.n) * p.m;
    for (int64_t t = tid; t < count; t += stride) {
      const int64_t j = t / p.n, i = t - j * p.n;
      const float v = __half2float(__ushort_as_half(__ldcg(p.B + j * p.ldb + i)));
      p.X[j * p.ldx + i] = __half_as_ushort(__float2half_rn(p.alpha * v));
    }
  }
}

// The previous values of columns [col, col + 32) of row `row` of Xᵀ, when
// all 32 lie before n_end (else zeros: store32 then reads them one by one).
__device__ __forceinline__ void load_old32(const ChainArgs& p, int64_t row, int col, int n_end, uint4 (&old)[4]) {
  const uint16_t* src = p.X + row * p.ldx + col;
  if (col + 32 <= n_end && HG_DBG_ALIGN(src, 16)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) old[j] = __ldcg(reinterpret_cast<const uint4*>(src) + j);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) old[j] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The epilogue of 32 columns [col, col + 32) of row `row` of Xᵀ: products
// store the accumulator, updates the previous value (`old`, from load_old32)
// minus it (one FP32 subtraction, one rounding). Columns at or past n_end
// are left alone.
__device__ __forceinline__ void store32(const ChainArgs& p, int kind, int64_t row, int col, int n_end,
                                        const uint32_t (&v)[32], const uint4 (&old)[4]) {
  uint16_t* dst = p.X + row * p.ldx + col;
  if (col + 32 <= n_end && HG_DBG_ALIGN(dst, 16)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      const __half* oh = reinterpret_cast<const __half*>(&old[j]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float acc = __uint_as_float(v[8 * j + i]);
        f[i] = kind == kChainUpdate ? __half2float(oh[i]) - acc : acc;
      }
      uint4 r;
      r.x = pack_half2(__float_as_uint(f[0]), __float_as_uint(f[1]));
      r.y = pack_half2(__float_as_uint(f[2]), __float_as_uint(f[3]));
      r.z = pack_half2(__float_as_uint(f[4]), __float_as_uint(f[5]));
      r.w = pack_half2(__float_as_uint(f[6]), __float_as_uint(f[7]));
      reinterpret_cast<uint4*>(dst)[j] = r;
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (col + i >= n_end) break;
    const float acc = __uint_as_float(v[i]);
    const float f = kind == kChainUpdate ? __half2float(__ushort_as_half(__ldcg(dst + i))) - acc : acc;
    dst[i] = __half_as_ushort(__float2half_rn(f));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    trsm_chain_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmWr, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ ChainArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar0 = ring + kOffBar;
  const uint32_t drain_bar = bar0 + 8 * (2 * kMaxStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile uint32_t* passed = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 8);  // grid barriers passed
  volatile int* epi_ok = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  ChainPhase* phases = reinterpret_cast<ChainPhase*>(smem + kOffPhases);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int num_phases = p.num_phases;

  // The phase table, read once from the parameters (reads of a new entry
  // there at every phase would each wait on the constant cache).
  for (int i = threadIdx.x; i < num_phases; i += blockDim.x) phases[i] = p.phase[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full_bar(s), 1);   // the producer's arrive.expect_tx (+ TMA bytes)
      mbar_init(empty_bar(s), 1);  // the MMA issuer's tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);  // tcgen05.commit after a tile
      mbar_init(acce_bar(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *passed = 0u;
    *epi_ok = 1;
    fence_barrier_init();
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmWr);
    prefetch_tensormap(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // the inverses, the synchronisation words and X come from the previous
  // launches on the stream
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // bit s of ebits: parity of the next wait on empty[s] (1 before stage s
      // is first filled), which is also the parity of full[s]'s phase that
      // its last fill completes; filled: stages filled at least once
      uint32_t ebits = 0xFFFFFFFFu, filled = 0u;
      long long fills = 0;
      int pref = 0;        // stages of this phase's first tile whose B boxes are already in flight
      bool ok = true;
      int j = 0;
      for (; j < num_phases && ok; ++j) {
        const Phase ph = decode(phases[j], p.m);
        if (j > 0) {
          // grid barrier j passed: the other CTAs' writes of X are visible,
          // and ordered before this thread's TMA reads
          ok = wait_passed(passed, static_cast<uint32_t>(j), wd);
          if (!ok) break;
          fence_proxy_async_global();
        }
        if (ph.kind != kChainCopy) {
          const CUtensorMap* mb = map_b(ph, &tmW, &tmWr, &tmA);
          int s = 0;
          bool first = true;
          for (int t = blockIdx.x; ok && t < ph.num_tiles; t += gridDim.x) {
            int mi, ni;
            tile_of(ph, t, mi, ni);
            for (int kk = 0; kk < ph.ksteps; ++kk) {
              const uint32_t sa = ring + s * ph.stage_bytes;
              if (!(first && kk < pref)) {
                if (!wait_phase(empty_bar(s), (ebits >> s) & 1u, wd, kWdProducerEmpty)) {
                  ok = false;
                  break;
                }
                ebits ^= 1u << s;
                filled |= 1u << s;
                if (!(p.inject == 1 && fills == 0))  // testing aid: withhold one arrival
                  mbar_arrive_expect_tx(full_bar(s), ph.tx_bytes);
                ++fills;
                load_b(ph, mb, sa + kASlot, full_bar(s), ni, kk);
              }
              load_a(ph, &tmX, sa, full_bar(s), mi, kk);
              if (++s == ph.stages) s = 0;
            }
            first = false;
          }
        }
        pref = 0;
        // The next phase's first stages of the second operand (which no
        // phase writes), before its barrier. The ring's geometry may change
        // with the phase, so every stage of this one must be consumed first.
        if (ok && j + 1 < num_phases) {
          const Phase nx = decode(phases[j + 1], p.m);
          if (nx.kind != kChainCopy && static_cast<int>(blockIdx.x) < nx.num_tiles) {
            for (int s2 = 0; s2 < kMaxStages && ok; ++s2)
              ok = wait_phase(empty_bar(s2), (ebits >> s2) & 1u, wd, kWdProducerEmpty);
            int mi, ni;
            tile_of(nx, blockIdx.x, mi, ni);
            const CUtensorMap* nmb = map_b(nx, &tmW, &tmWr, &tmA);
            const int np = min(nx.ksteps, nx.stages);
            for (int kk = 0; ok && kk < np; ++kk) {
              ebits ^= 1u << kk;
              filled |= 1u << kk;
              if (!(p.inject == 1 && fills == 0)) mbar_arrive_expect_tx(full_bar(kk), nx.tx_bytes);
              ++fills;
              load_b(nx, nmb, ring + kk * nx.stage_bytes + kASlot, full_bar(kk), ni, kk);
              pref = kk + 1;
            }
          }
        }
      }
      // Stages whose B boxes went out before an aborted barrier still expect
      // their Xᵀ bytes: issue those loads (phase j), then wait until every
      // fill has landed.
      if (pref > 0 && j < num_phases) {
        const Phase nx = decode(phases[j], p.m);
        int mi, ni;
        tile_of(nx, blockIdx.x, mi, ni);
        for (int kk = 0; kk < pref; ++kk) load_a(nx, &tmX, ring + kk * nx.stage_bytes, full_bar(kk), mi, kk);
      }
      for (int s = 0; s < kMaxStages; ++s)
        if ((filled >> s) & 1u) wait_drain(full_bar(s), (ebits >> s) & 1u, wd);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t fbits = 0;  // parity of the next wait on full[s]
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int j = 0; j < num_phases && ok; ++j) {
        const Phase ph = decode(phases[j], p.m);
        if (ph.kind == kChainCopy) continue;
        const uint32_t idesc = idesc_f16_f32acc(kTcBM, ph.bn) | idesc_major_bits(false, ph.b_mn != 0);
        const uint32_t b_step = ph.b_mn ? 128u : 2u;  // 16 K: 16 rows of 128 B, or 32 B along the row
        int s = 0;
        for (int t = blockIdx.x; ok && t < ph.num_tiles; t += gridDim.x) {
          int mi, ni;
          tile_of(ph, t, mi, ni);
          if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
          for (int kk = 0; kk < ph.ksteps; ++kk) {
            if (!wait_phase(full_bar(s), (fbits >> s) & 1u, wd, kWdMmaFull)) {
              ok = false;
              break;
            }
            fbits ^= 1u << s;
            if (ph.kind == kChainProduct && kk == ph.ksteps - 1) {
              // every Xᵀ box of this tile has landed: its reads of the rows are done
              const int g0 = mi * ph.bm / 64;
              for (int g = g0; g < g0 + ph.bm / 64 && g < kChainMaxRowGroups; ++g)
                red_relaxed_gpu(p.sync + kChainSyncRowGroup0 + g, 1u);
            }
            tc_fence_after_sync();
            const uint32_t sa = ring + s * ph.stage_bytes;
            const uint64_t a_desc = sdesc_kmajor_sw128(sa);
            const uint64_t b_desc = ph.b_mn ? sdesc_mnmajor_sw128(sa + kASlot) : sdesc_kmajor_sw128(sa + kASlot);
#pragma unroll
            for (int k = 0; k < kTcBK / 16; ++k)
              mma_f16_ss(d_tmem, a_desc + 2u * k, b_desc + b_step * k, idesc, (kk > 0 || k > 0) ? 1u : 0u);
            mma_commit(empty_bar(s));
            if (++s == ph.stages) s = 0;
          }
          if (!ok) break;
          mma_commit(accf_bar(acc));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      mma_commit(drain_bar);  // every MMA issued above completes before TMEM is freed
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- epilogue (warps 2–5)
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 = tile rows of this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int j = 0; j < num_phases && ok; ++j) {
      const Phase ph = decode(phases[j], p.m);
      if (ph.kind == kChainCopy) copy_phase(p);
      for (int t = blockIdx.x; ok && t < ph.num_tiles; t += gridDim.x) {
        int mi, ni;
        tile_of(ph, t, mi, ni);
        const int r0 = mi * ph.bm + 32 * q;  // this warp's first row
        const bool rows = 32 * q < ph.bm && r0 < p.m;
        const int64_t row = static_cast<int64_t>(r0) + lane;
        const int c0 = ph.n0 + ni * ph.bn;
        const bool upd = ph.kind == kChainUpdate;
        // updates: the first 32 previous values are read while the MMAs run
        uint4 old[4] = {};
        if (upd && rows && row < p.m) load_old32(p, row, c0, ph.n_end, old);
        int good = 1;
        if (lane == 0) {
          if (ph.kind == kChainProduct && rows) {
            // the other tiles of these rows must have read them
            const uint32_t* ctr = p.sync + kChainSyncRowGroup0 + r0 / 64;
            if (ld_relaxed_gpu(ctr) < ph.rg_target) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_relaxed_gpu(ctr) < ph.rg_target) {
                if (*abort_flag || launch_aborted(p)) {
                  *abort_flag = 1;
                  good = 0;
                  break;
                }
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                  wd.raise(kWdRowGroup);
                  good = 0;
                  break;
                }
              }
            }
          }
          if (good) good = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (rows) {
          const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                 static_cast<uint32_t>(acc * kAccCols);
#pragma unroll 1
          for (int c = 0; c < ph.bn / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + 32 * c, v);
            // the next chunk's previous values, in flight during this one
            uint4 nxt[4] = {};
            if (upd && row < p.m && c + 1 < ph.bn / 32) load_old32(p, row, c0 + 32 * (c + 1), ph.n_end, nxt);
            tmem_ld_wait(v);
            if (row < p.m && c0 + 32 * c < ph.n_end) store32(p, ph.kind, row, c0 + 32 * c, ph.n_end, v, old);
#pragma unroll
            for (int i = 0; i < 4; ++i) old[i] = nxt[i];
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // A role that gave up raised the CTA's abort flag; the barrier spreads
      // it (every epilogue warp calls it, whether its own tiles went well or
      // not, and all four take the leader's verdict).
      if (j + 1 < num_phases) ok = grid_barrier(p, static_cast<uint32_t>(j) + 1u, abort_flag, passed, epi_ok);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

constexpr int kMaxDevices = 64;

}  // namespace

int chain_max_grid(int num_sms) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cached[dev] > 0) return cached[dev];
  int per_sm = 0;
  if (cudaFuncSetAttribute(trsm_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, trsm_chain_kernel, kThreads, kSmemBytes) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const int g = per_sm >= 1 ? num_sms : 0;  // one CTA per SM: TMEM and the ring take the SM
  cached[dev] = g;
  return g;
}

cudaError_t launch_trsm_chain(const CUtensorMap& x, const CUtensorMap& w, const CUtensorMap& wr,
                              const CUtensorMap& a, const ChainArgs& args, int grid, cudaStream_t stream) {
  if (grid < 1 || args.num_phases < 1 || args.num_phases > kChainMaxPhases) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> attr_done[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev]) {
    e = cudaFuncSetAttribute(trsm_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev] = true;
  }
  // Cooperative: every CTA is resident at once (or the launch fails), which
  // the grid barriers need. With programmatic stream serialization its
  // launch and prologue overlap the inverses' launch, whose completion it
  // waits for (griddepcontrol.wait) before touching memory; where the two
  // attributes cannot be combined, it is launched without the overlap.
  static std::atomic<int> pdl_ok[kMaxDevices];  // 0 untried, 1 combined launches work, -1 they fail
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (!known || pdl_ok[dev] >= 0) {
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, trsm_chain_kernel, x, w, wr, a, args);
    if (e == cudaSuccess) {
      if (known) pdl_ok[dev] = 1;
      return e;
    }
    if (!known || pdl_ok[dev] == 1) return e;
    (void)cudaGetLastError();  // the combination is refused before anything is enqueued
    pdl_ok[dev] = -1;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, trsm_chain_kernel, x, w, wr, a, args);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(chain)

}  // namespace hg
