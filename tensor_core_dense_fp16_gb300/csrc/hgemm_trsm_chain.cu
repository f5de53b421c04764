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
//   * X := alpha·B is folded into the first phase that reads each block:
//     the first product takes its first operand from B and scales its
//     accumulator by alpha, the first update subtracts from alpha·B (one
//     FP32 product and one rounding per element). Only when B does not suit
//     TMA is a copy phase (grid-stride, by the epilogue warps) run first;
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
#include "trsm_chain.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

constexpr int kThreads = 192;                     // producer, MMA issuer, four epilogue warps
constexpr int kRingBytes = 192 * 1024;            // operand ring, regrouped into stages per tile shape
constexpr int kMaxStages = 8;
constexpr int kASlot = kTcBM * kTcBK * 2;         // 16 KB: an M=128 MMA reads 128 rows
constexpr int kBox = 64;                          // every TMA box is 64 × 64 elements
constexpr int kBoxBytes = kBox * kBox * 2;        // 8 KB
constexpr int kAccCols = 256;                     // the widest tile: 256 FP32 columns
constexpr int kTmemCols = 2 * kAccCols;           // two accumulators
constexpr int kSlot = kTrsmInverseLeaf;           // rows and columns of a workspace slot
constexpr int kOffBar = kRingBytes;
// full, empty, accumulator full ×2 / empty ×2, drain
constexpr int kNumBars = 2 * kMaxStages + 4 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM address, abort flag, barriers passed, epilogue verdict
constexpr int kOffGroups = kOffMisc + 16;         // the group table, decoded from the parameters
constexpr int kEpiThreads = 128;                  // warps 2–5
constexpr int kEpiBarrier = 1;                    // named barrier of the epilogue warps
static_assert(kRingBytes / (kASlot + 64 * kTcBK * 2) >= kMaxStages, "the narrowest stages fill the ring");
static_assert(5 * sizeof(CUtensorMap) + sizeof(ChainArgs) <= 4096, "kernel parameters beyond 4 KB");

// A group, decoded.
struct Group {
  int kind, a_map, a_mn, b_map, b_mn, bm, bn, old_from_b, last, critical;
  int rows, n0, n_end;
  int a_kbase, a_mbase, ksteps, b_kbase, b_nbase, a2_kbase, b2_kbase, ksteps2, out_slot;
  float scale;
  uint32_t rg_target;
  int num_m, num_n, tiles;
  uint32_t stage_bytes, tx_bytes;
  int stages;
};
constexpr int kSmemBytes = kOffGroups + kChainMaxGroups * static_cast<int>(sizeof(Group)) + 1024;
static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory per CTA");

__device__ __forceinline__ Group decode(const ChainGroup& c) {
  Group g;
  g.kind = c.flags & 3u;
  g.a_map = (c.flags >> 2) & 7u;
  g.a_mn = (c.flags >> 5) & 1u;
  g.b_map = (c.flags >> 6) & 7u;
  g.b_mn = (c.flags >> 9) & 1u;
  g.bm = ((c.flags >> 10) & 3u) * 64;
  g.bn = ((c.flags >> 12) & 7u) * 64;
  g.old_from_b = (c.flags >> 15) & 1u;
  g.last = (c.flags >> 16) & 1u;
  g.critical = (c.flags >> 17) & 1u;
  g.rows = c.rows;
  g.n0 = c.n0;
  g.n_end = c.n_end;
  g.a_kbase = c.a_kbase;
  g.a_mbase = c.a_mbase;
  g.ksteps = c.ksteps;
  g.b_kbase = c.b_kbase;
  g.b_nbase = c.b_nbase;
  g.a2_kbase = c.a2_kbase;
  g.b2_kbase = c.b2_kbase;
  g.ksteps2 = c.ksteps2;
  g.out_slot = c.out_slot;
  g.scale = c.scale;
  g.rg_target = c.rg_target;
  if (g.kind == kChainCopy || g.bm == 0 || g.bn == 0) {
    g.num_m = g.num_n = g.tiles = 0;
    g.stages = 1;
    g.stage_bytes = g.tx_bytes = 0;
    return g;
  }
  g.num_m = (g.rows + g.bm - 1) / g.bm;
  g.num_n = (g.n_end - g.n0 + g.bn - 1) / g.bn;
  g.tiles = g.num_m * g.num_n;
  g.stage_bytes = static_cast<uint32_t>(kASlot + g.bn * kTcBK * 2);
  g.stages = min(kMaxStages, static_cast<int>(kRingBytes / g.stage_bytes));
  g.tx_bytes = static_cast<uint32_t>((g.bm / kBox + g.bn / kBox) * kBoxBytes);
  return g;
}

// Tile t of a group: row tile mi, column tile ni (column-tile major, so that
// concurrently running tiles share the second operand's boxes).
__device__ __forceinline__ void tile_of(const Group& g, int t, int& mi, int& ni) {
  ni = t / g.num_m;
  mi = t - ni * g.num_m;
}

// One unit of work of a CTA: a group index and a tile of it.
struct Task {
  int group, tile;
};

// The tasks of CTA `cta` (of `ctas`) in the phase whose groups are [g0, g1]:
// the critical group's tiles (the products) one per CTA on CTAs [0, P), then
// the other groups' tiles, concatenated, round-robin over CTAs [P, ctas)
// (over all CTAs when P fills the grid). Task i of the CTA, or group -1.
__device__ __forceinline__ Task task_at(const Group* groups, int g0, int g1, int cta, int ctas, int i) {
  const Group& first = groups[g0];
  const int crit = first.critical ? first.tiles : 0;
  if (cta < crit) {
    if (i == 0) return Task{g0, cta};
    --i;
  }
  const int lo = crit < ctas ? crit : 0;  // the CTAs that take the other groups
  if (cta < lo) return Task{-1, 0};
  const int span = ctas - lo;
  int idx = (cta - lo) + i * span;
  for (int g = first.critical ? g0 + 1 : g0; g <= g1; ++g) {
    const int n = groups[g].tiles;
    if (idx < n) return Task{g, idx};
    idx -= n;
  }
  return Task{-1, 0};
}

// The last group of the phase that starts at group g0.
__device__ __forceinline__ int phase_end(const Group* groups, int g0, int num_groups) {
  int g = g0;
  while (g + 1 < num_groups && !groups[g].last) ++g;
  return g;
}

__device__ __forceinline__ const CUtensorMap* map_of(int which, const CUtensorMap* x, const CUtensorMap* b,
                                                     const CUtensorMap* w, const CUtensorMap* wr,
                                                     const CUtensorMap* a) {
  return which == kChainMapX ? x : which == kChainMapB ? b : which == kChainMapW ? w : which == kChainMapWRagged ? wr : a;
}

// Operand boxes of k-step kk (of both segments) of tile (mi, ni) into the
// stage at `sa` (first operand) and `sa + kASlot` (second operand).
// b_only / a_only: one operand (the second is prefetched before a barrier).
struct Maps {
  const CUtensorMap *x, *b, *w, *wr, *a;
};

__device__ __forceinline__ void load_b(const Group& g, const Maps& m, uint32_t sb, uint32_t bar, int ni, int kk) {
  const bool seg2 = kk >= g.ksteps;
  const CUtensorMap* map = seg2 ? m.w : map_of(g.b_map, m.x, m.b, m.w, m.wr, m.a);
  const int kc = seg2 ? g.b2_kbase + (kk - g.ksteps) * kTcBK : g.b_kbase + kk * kTcBK;
  const int nb = seg2 ? 0 : g.b_nbase;
  const bool mn = seg2 || g.b_mn;
  for (int i = 0; i < g.bn / kBox; ++i) {
    const int nc = nb + ni * g.bn + i * kBox;
    if (mn)
      tma_load_2d(sb + i * kBoxBytes, map, bar, nc, kc);  // box: 64 N (contiguous) × 64 K rows
    else
      tma_load_2d(sb + i * kBoxBytes, map, bar, kc, nc);  // box: 64 N rows × 64 K (contiguous)
  }
}

__device__ __forceinline__ void load_a(const Group& g, const Maps& m, uint32_t sa, uint32_t bar, int mi, int kk) {
  const bool seg2 = kk >= g.ksteps;
  const CUtensorMap* map = seg2 ? m.x : map_of(g.a_map, m.x, m.b, m.w, m.wr, m.a);
  const int kc = seg2 ? g.a2_kbase + (kk - g.ksteps) * kTcBK : g.a_kbase + kk * kTcBK;
  const bool mn = !seg2 && g.a_mn;
  for (int i = 0; i < g.bm / kBox; ++i) {
    const int mc = (seg2 ? 0 : g.a_mbase) + mi * g.bm + i * kBox;
    if (mn)
      tma_load_2d(sa + i * kBoxBytes, map, bar, mc, kc);  // box: 64 M (contiguous) × 64 K rows
    else
      tma_load_2d(sa + i * kBoxBytes, map, bar, kc, mc);  // box: 64 M rows × 64 K (contiguous)
  }
}

// The TMA boxes of one operand over one K segment of a task, worked out
// once per task so that the producer's per-step work is a few additions and
// the copies: box i of the segment's k-step kk is at
// (x0 + kk·kdx + i·bdx, y0 + kk·kdy + i·bdy) of `map`.
struct OperandStream {
  const CUtensorMap* map;
  int x0, y0, kdx, kdy, bdx, bdy, boxes;
};

// The coordinates load_a and load_b use, as streams: the first operand of
// segment `seg2` (0: the task's first K segment) for row tile mi, the second
// for column tile ni.
__device__ __forceinline__ OperandStream stream_a(const Group& g, const Maps& m, int mi, bool seg2) {
  const bool mn = !seg2 && g.a_mn;
  const int kc0 = seg2 ? g.a2_kbase : g.a_kbase;
  const int mc0 = (seg2 ? 0 : g.a_mbase) + mi * g.bm;
  OperandStream o;
  o.map = seg2 ? m.x : map_of(g.a_map, m.x, m.b, m.w, m.wr, m.a);
  o.boxes = g.bm / kBox;
  if (mn) {
    o.x0 = mc0, o.y0 = kc0, o.kdx = 0, o.kdy = kTcBK, o.bdx = kBox, o.bdy = 0;
  } else {
    o.x0 = kc0, o.y0 = mc0, o.kdx = kTcBK, o.kdy = 0, o.bdx = 0, o.bdy = kBox;
  }
  return o;
}
__device__ __forceinline__ OperandStream stream_b(const Group& g, const Maps& m, int ni, bool seg2) {
  const bool mn = seg2 || g.b_mn;
  const int kc0 = seg2 ? g.b2_kbase : g.b_kbase;
  const int nc0 = (seg2 ? 0 : g.b_nbase) + ni * g.bn;
  OperandStream o;
  o.map = seg2 ? m.w : map_of(g.b_map, m.x, m.b, m.w, m.wr, m.a);
  o.boxes = g.bn / kBox;
  if (mn) {
    o.x0 = nc0, o.y0 = kc0, o.kdx = 0, o.kdy = kTcBK, o.bdx = kBox, o.bdy = 0;
  } else {
    o.x0 = kc0, o.y0 = nc0, o.kdx = kTcBK, o.kdy = 0, o.bdx = 0, o.bdy = kBox;
  }
  return o;
}
__device__ __forceinline__ void load_stream(const OperandStream& o, uint32_t dst, uint32_t bar, int kk) {
  const int x = o.x0 + kk * o.kdx, y = o.y0 + kk * o.kdy;
  tma_load_2d(dst, o.map, bar, x, y);
  for (int i = 1; i < o.boxes; ++i) tma_load_2d(dst + i * kBoxBytes, o.map, bar, x + i * o.bdx, y + i * o.bdy);
}

// True once the phase with parity `parity` of `bar` has completed, without
// suspending (a stage that landed during the previous stage's MMAs is then
// taken at once; otherwise the caller falls back to the suspending wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  if (!HG_DBG_SMEM(bar, 8)) return false;
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
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

// The previous values of columns [col, col + 32) of row `row` of Xᵀ (from_b:
// of Bᵀ), when all 32 lie before n_end (else zeros: store32 then reads them
// one by one).
__device__ __forceinline__ void load_old32(const ChainArgs& p, bool from_b, int64_t row, int col, int n_end,
                                           uint4 (&old)[4]) {
  const uint16_t* src = from_b ? p.B + row * p.ldb + col : p.X + row * p.ldx + col;
  if (col + 32 <= n_end && HG_DBG_ALIGN(src, 16)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) old[j] = __ldcg(reinterpret_cast<const uint4*>(src) + j);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) old[j] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The epilogue of 32 columns [col, col + 32) of row `row`: updates store the
// previous value (`old`, from load_old32; alpha·B when from_b) minus the
// accumulator (one FP32 operation, one rounding), products and couplings
// scale · acc, into `dst` (the row's element `col`). Columns at or past
// n_end are left alone.
__device__ __forceinline__ void store32(const ChainArgs& p, bool update, bool from_b, float scale, uint16_t* dst,
                                        const uint16_t* src_old, int col, int n_end, const uint32_t (&v)[32],
                                        const uint4 (&old)[4]) {
  const float oscale = from_b ? p.alpha : 1.0f;
  if (col + 32 <= n_end && HG_DBG_ALIGN(dst, 16)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      const __half* oh = reinterpret_cast<const __half*>(&old[j]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float acc = __uint_as_float(v[8 * j + i]);
        f[i] = update ? oscale * __half2float(oh[i]) - acc : scale * acc;
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
    const float f = update ? oscale * __half2float(__ushort_as_half(__ldcg(src_old + i))) - acc : scale * acc;
    dst[i] = __half_as_ushort(__float2half_rn(f));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    trsm_chain_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWr,
                      const __grid_constant__ CUtensorMap tmA, const __grid_constant__ ChainArgs p) {
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
  Group* groups = reinterpret_cast<Group*>(smem + kOffGroups);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int num_groups = p.num_groups;
  const int cta = static_cast<int>(blockIdx.x), ctas = static_cast<int>(gridDim.x);
  const Maps maps{&tmX, &tmB, &tmW, &tmWr, &tmA};

  // The group table, read once from the parameters and decoded (reads of a
  // new entry there at every phase would each wait on the constant cache).
  for (int i = threadIdx.x; i < num_groups; i += blockDim.x) groups[i] = decode(p.group[i]);
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
    prefetch_tensormap(&tmB);
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
      uint32_t cur_sb = 0;  // the ring's current stage size (0: none yet)
      int s = 0;            // next stage
      int pref = 0;         // stages of the phase's first task whose second operand is already in flight
      int pref_group = -1, pref_tile = 0;
      bool ok = true;
      int j = 0, g0 = 0;
      // every stage consumed, then the ring regrouped for stages of sb bytes
      auto regroup = [&](uint32_t sb) {
        for (int s2 = 0; s2 < kMaxStages && ok; ++s2)
          ok = wait_phase(empty_bar(s2), (ebits >> s2) & 1u, wd, kWdProducerEmpty);
        cur_sb = sb;
        s = 0;
      };
      for (; g0 < num_groups && ok; ++j) {
        const int g1 = phase_end(groups, g0, num_groups);
        if (j > 0) {
          // grid barrier j passed: the other CTAs' writes are visible, and
          // ordered before this thread's TMA reads
          ok = wait_passed(passed, static_cast<uint32_t>(j), wd);
          if (!ok) break;
          fence_proxy_async_global();
        }
        for (int i = 0; ok; ++i) {
          const Task tk = task_at(groups, g0, g1, cta, ctas, i);
          if (tk.group < 0) break;
          const Group g = groups[tk.group];  // a copy: the loops below read it from registers
          if (g.kind == kChainCopy) continue;
          const bool prefetched = i == 0 && pref > 0;
          if (!prefetched && g.stage_bytes != cur_sb) regroup(g.stage_bytes);
          int mi, ni;
          tile_of(g, tk.tile, mi, ni);
          const int kall = g.ksteps + g.ksteps2;
          const OperandStream a1 = stream_a(g, maps, mi, false), a2 = stream_a(g, maps, mi, true);
          const OperandStream b1 = stream_b(g, maps, ni, false), b2 = stream_b(g, maps, ni, true);
          for (int kk = 0; ok && kk < kall; ++kk) {
            const uint32_t sa = ring + s * g.stage_bytes;
            const bool seg2 = kk >= g.ksteps;
            const int kl = seg2 ? kk - g.ksteps : kk;
            if (!(prefetched && kk < pref)) {
              // a stage freed during the previous copies is taken without suspending
              if (!mbar_test_wait(empty_bar(s), (ebits >> s) & 1u) &&
                  !wait_phase(empty_bar(s), (ebits >> s) & 1u, wd, kWdProducerEmpty)) {
                ok = false;
                break;
              }
              ebits ^= 1u << s;
              filled |= 1u << s;
              if (!(p.inject == 1 && fills == 0))  // testing aid: withhold one arrival
                mbar_arrive_expect_tx(full_bar(s), g.tx_bytes);
              ++fills;
              load_stream(seg2 ? b2 : b1, sa + kASlot, full_bar(s), kl);
            }
            load_stream(seg2 ? a2 : a1, sa, full_bar(s), kl);
            if (++s == g.stages) s = 0;
          }
        }
        pref = 0;
        pref_group = -1;
        // The next phase's first task: the stages of its first K segment
        // take their second operand (an inverse or the triangle, which no
        // phase writes while it is still to be read) before the barrier.
        const int n0g = g1 + 1;
        if (ok && n0g < num_groups) {
          const int n1g = phase_end(groups, n0g, num_groups);
          const Task tk = task_at(groups, n0g, n1g, cta, ctas, 0);
          if (tk.group >= 0) {
            const Group g = groups[tk.group];  // a copy: the loops below read it from registers
            if (g.kind != kChainCopy) {
              regroup(g.stage_bytes);
              int mi, ni;
              tile_of(g, tk.tile, mi, ni);
              const int np = min(g.ksteps, g.stages);
              pref_group = tk.group;
              pref_tile = tk.tile;
              for (int kk = 0; ok && kk < np; ++kk) {
                ebits ^= 1u << kk;
                filled |= 1u << kk;
                if (!(p.inject == 1 && fills == 0)) mbar_arrive_expect_tx(full_bar(kk), g.tx_bytes);
                ++fills;
                load_b(g, maps, ring + kk * g.stage_bytes + kASlot, full_bar(kk), ni, kk);
                pref = kk + 1;
              }
            }
          }
        }
        g0 = g1 + 1;
      }
      // Stages whose second operand went out before an aborted barrier still
      // expect their Xᵀ bytes: issue those loads, then wait until every fill
      // has landed.
      if (pref > 0 && pref_group >= 0) {
        const Group g = groups[pref_group];
        int mi, ni;
        tile_of(g, pref_tile, mi, ni);
        for (int kk = 0; kk < pref; ++kk) load_a(g, maps, ring + kk * g.stage_bytes, full_bar(kk), mi, kk);
      }
      for (int s2 = 0; s2 < kMaxStages; ++s2)
        if ((filled >> s2) & 1u) wait_drain(full_bar(s2), (ebits >> s2) & 1u, wd);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t fbits = 0;  // parity of the next wait on full[s]
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t cur_sb = 0;
      int s = 0;
      bool ok = true;
      for (int g0 = 0; g0 < num_groups && ok;) {
        const int g1 = phase_end(groups, g0, num_groups);
        for (int i = 0; ok; ++i) {
          const Task tk = task_at(groups, g0, g1, cta, ctas, i);
          if (tk.group < 0) break;
          const Group g = groups[tk.group];  // a copy: the loops below read it from registers
          if (g.kind == kChainCopy) continue;
          // the producer regroups the ring at the same points
          if (g.stage_bytes != cur_sb) {
            cur_sb = g.stage_bytes;
            s = 0;
          }
          // prefetched first tasks start on stage 0 as well
          if (i == 0) s = 0;
          int mi, ni;
          tile_of(g, tk.tile, mi, ni);
          if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
          const int kall = g.ksteps + g.ksteps2;
          for (int kk = 0; kk < kall; ++kk) {
            if (!mbar_test_wait(full_bar(s), (fbits >> s) & 1u) &&
                !wait_phase(full_bar(s), (fbits >> s) & 1u, wd, kWdMmaFull)) {
              ok = false;
              break;
            }
            fbits ^= 1u << s;
            if (g.critical && kk == kall - 1) {
              // every Xᵀ box of this product tile has landed: its reads of the rows are done
              const int r0 = mi * g.bm / 64;
              for (int r = r0; r < r0 + g.bm / 64 && r < kChainMaxRowGroups; ++r)
                red_relaxed_gpu(p.sync + kChainSyncRowGroup0 + r, 1u);
            }
            tc_fence_after_sync();
            const bool seg2 = kk >= g.ksteps;
            const bool amn = !seg2 && g.a_mn, bmn = seg2 || g.b_mn;
            const uint32_t idesc = idesc_f16_f32acc(kTcBM, g.bn) | idesc_major_bits(amn, bmn);
            const uint32_t sa = ring + s * g.stage_bytes;
            const uint64_t a_desc = amn ? sdesc_mnmajor_sw128(sa) : sdesc_kmajor_sw128(sa);
            const uint64_t b_desc = bmn ? sdesc_mnmajor_sw128(sa + kASlot) : sdesc_kmajor_sw128(sa + kASlot);
            // 16 K: 16 rows of 128 B (N/M-contiguous), or 32 B along the row
            const uint32_t a_step = amn ? 128u : 2u, b_step = bmn ? 128u : 2u;
#pragma unroll
            for (int k = 0; k < kTcBK / 16; ++k)
              mma_f16_ss(d_tmem, a_desc + a_step * k, b_desc + b_step * k, idesc, (kk > 0 || k > 0) ? 1u : 0u);
            mma_commit(empty_bar(s));
            if (++s == g.stages) s = 0;
          }
          if (!ok) break;
          mma_commit(accf_bar(acc));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        g0 = g1 + 1;
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
    uint32_t barrier = 0;
    for (int g0 = 0; g0 < num_groups && ok;) {
      const int g1 = phase_end(groups, g0, num_groups);
      if (groups[g0].kind == kChainCopy) copy_phase(p);
      for (int i = 0; ok; ++i) {
        const Task tk = task_at(groups, g0, g1, cta, ctas, i);
        if (tk.group < 0) break;
        const Group g = groups[tk.group];  // a copy: the loops below read it from registers
        if (g.kind == kChainCopy) continue;
        int mi, ni;
        tile_of(g, tk.tile, mi, ni);
        const bool coupling = g.kind == kChainCoupling, upd = g.kind == kChainUpdate;
        const int r0 = mi * g.bm + 32 * q;  // this warp's first row
        const int row_lim = coupling ? kSlot : g.rows;
        const bool rows = 32 * q < g.bm && r0 < row_lim;
        const int64_t row = static_cast<int64_t>(r0) + lane;
        const int c0 = g.n0 + ni * g.bn;
        const bool from_b = g.old_from_b != 0;
        // updates: the previous values of the first 64 columns (a 64-column
        // tile's all) are read while the MMAs run
        uint4 old[4] = {}, old2[4] = {};
        if (upd && rows && row < row_lim) {
          load_old32(p, from_b, row, c0, g.n_end, old);
          load_old32(p, from_b, row, c0 + 32, g.n_end, old2);
        }
        int good = 1;
        if (lane == 0) {
          if (g.critical && rows) {
            // the other tiles of these rows must have read them
            const uint32_t* ctr = p.sync + kChainSyncRowGroup0 + r0 / 64;
            if (ld_relaxed_gpu(ctr) < g.rg_target) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_relaxed_gpu(ctr) < g.rg_target) {
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
          uint16_t* drow = coupling ? p.W + static_cast<int64_t>(g.out_slot) * kSlot * kSlot + row * kSlot
                                    : p.X + row * p.ldx;
          const uint16_t* orow = from_b ? p.B + row * p.ldb : p.X + row * p.ldx;
#pragma unroll 1
          for (int c = 0; c < g.bn / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + 32 * c, v);
            // the previous values two chunks ahead, in flight during this one
            uint4 nxt[4] = {};
            if (upd && row < row_lim && c + 2 < g.bn / 32) load_old32(p, from_b, row, c0 + 32 * (c + 2), g.n_end, nxt);
            tmem_ld_wait(v);
            const int col = c0 + 32 * c;
            if (row < row_lim && col < g.n_end)
              store32(p, upd, from_b, g.scale, drow + col, orow + col, col, g.n_end, v, old);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              old[k] = old2[k];
              old2[k] = nxt[k];
            }
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
      g0 = g1 + 1;
      if (g0 < num_groups) ok = grid_barrier(p, ++barrier, abort_flag, passed, epi_ok);
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

cudaError_t launch_trsm_chain(const CUtensorMap& x, const CUtensorMap& b, const CUtensorMap& w,
                              const CUtensorMap& wr, const CUtensorMap& a, const ChainArgs& args, int grid,
                              cudaStream_t stream) {
  if (grid < 1 || args.num_groups < 1 || args.num_groups > kChainMaxGroups) return cudaErrorInvalidValue;
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
    e = cudaLaunchKernelEx(&cfg, trsm_chain_kernel, x, b, w, wr, a, args);
    if (e == cudaSuccess) {
      if (known) pdl_ok[dev] = 1;
      return e;
    }
    if (!known || pdl_ok[dev] == 1) return e;
    (void)cudaGetLastError();  // the combination is refused before anything is enqueued
    pdl_ok[dev] = -1;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, trsm_chain_kernel, x, b, w, wr, a, args);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(chain)

}  // namespace hg
