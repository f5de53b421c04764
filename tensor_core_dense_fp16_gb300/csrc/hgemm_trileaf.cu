// hgemm_trileaf.cu — the diagonal blocks ("leaves") of the recursive
// triangular product of "异构计算中高性能TRMM与TRSM的递归算法实现" (§2.1–§2.2:
// the recursion stops at diagonal blocks of order 256, which are multiplied
// directly) on the tensor cores.
//
// In the GEMM view of that product (Cᵀ = Bᵀ·lower(A), both operands
// K-contiguous; see hgemm_trmm), leaf b at offset `off` and of order s
// computes
//   Ct[:, off : off+s] = alpha · X[:, off : off+s] · L_b
// with X = Bᵀ (m × n, row pitch ldb), Ct = Cᵀ (m × n, row pitch ldc) and L_b
// the s × s operand whose row i is column off+i of A from row off on:
// L_b[i][k] = A(off+k, off+i) for k ≥ i, zero for k < i (A's strictly upper
// triangle is never used). This kernel takes leaves whose order is a multiple
// of 64 (every leaf when n is); the generic kernel takes the others.
//
// Design (one CTA per SM, tcgen05 with M = 128):
//   * persistent CTAs walk units (128-row tile of X, leaf), all leaves of one
//     tile consecutively (longest first), so the CTAs at work share those
//     rows of X, each read from memory once, while the leaves' operand rows
//     (A's lower part) stay in L2;
//   * a unit's 64-wide K blocks go in reverse order. K block kb meets only
//     rows i ≤ 64·kb + 63 of L_b (rows below are zero there), so TMA loads
//     just those 64·(kb + 1) rows and the MMA is N = 64·(kb + 1) wide: the
//     first (widest) block initialises all s accumulator columns, the later,
//     narrower ones accumulate into a prefix of them — 5/8 of the dense
//     product's MMA work for s = 256;
//   * rows i < 64·kb are whole in block kb; the 64×64 diagonal sub-block
//     (i = 64·kb + r, k = 64·kb + c) is masked in shared memory by the MMA
//     warp once its TMA copy has landed: elements with c < r are zeroed
//     before the MMAs read the stage;
//   * warp 0 streams the X tile and the triangle rows into a 4-stage ring;
//     the accumulator is double-buffered in TMEM (2 × 256 columns) and the
//     epilogue warps (TMEM → alpha·acc → FP16 round to nearest even →
//     swizzled staging → TMA store) drain one unit while the next one runs;
//   * a leaf may also carry the off-diagonal updates (C1 += alpha·A21ᵀ·B2 in
//     the page's recursion) of the small blocks whose first half holds it:
//     its product then runs on over K columns [off+s, off+s+ext) with whole
//     rows of the second operand (A21 lies below the diagonal), processed
//     first (N = s, initialising the accumulator), so those updates cost no
//     launch, no read-modify-write of C and no intermediate FP16 rounding;
//   * with few units (a short X), each unit's K blocks are split over a
//     cluster of CTAs instead, the partial sums reduced through distributed
//     shared memory (hgemm_tri_leaves_split_kernel below);
//   * every wait is bounded, as in the other tensor-core kernels (watchdog
//     word, abort flag, drain, TMEM freed).
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

struct LeafCfg {
  static constexpr int BM = kTcBM;                             // rows of X per unit
  static constexpr int BK = kTcBK;                             // K block
  static constexpr int MAX_S = 256;                            // widest leaf
  static constexpr int STAGES = 4;
  static constexpr int UMMA_K = 16;
  static constexpr int A_BYTES = BM * BK * 2;                  // X tile: 16 KB
  static constexpr int L_BOX_ROWS = 64;                        // triangle rows per TMA box
  static constexpr int L_BOX_BYTES = L_BOX_ROWS * BK * 2;      // 8 KB
  static constexpr int B_BYTES = MAX_S * BK * 2;               // up to 256 triangle rows: 32 KB
  static constexpr int EPI_WARPS = 4;
  static constexpr int C_BOX_BYTES = kEpiRows * kEpiCols * 2;  // 4 KB
  static constexpr int C_BUFS = 2;                             // per epilogue warp
  static constexpr int C_BYTES = EPI_WARPS * C_BUFS * C_BOX_BYTES;
  static constexpr int ACC_COLS = MAX_S;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;               // double buffer
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_C + C_BYTES;
  // full, empty, then: acc full/empty and drain (persistent kernel), or acc
  // full, drain, partials received and one "owner ready" per slice (split K)
  static constexpr int NUM_BARS = 2 * STAGES + 8;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;      // tmem address, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;      // + slack to align the base
  static constexpr int THREADS = 192;

  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && L_BOX_BYTES % 1024 == 0 &&
                    C_BOX_BYTES % 1024 == 0,
                "swizzled buffers must stay 1024-byte aligned");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
};

// Zeroes L(64kb + r, 64kb + c) for c < r in the 64×64 diagonal sub-block of
// a stage (128-byte-swizzled rows: the 16-byte chunk q of row r, elements
// c = 8q .. 8q+7, sits at chunk position q ^ (r % 8)). Lane l takes rows l
// and l + 32.
__device__ __forceinline__ void mask_diagonal_block(uint8_t* diag, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = lane + 32 * h;
    uint8_t* row = diag + r * 128;
    const int whole = r >> 3;  // chunks entirely left of the diagonal
    for (int q = 0; q < whole; ++q)
      *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    const int lead = r & 7;  // leading elements of chunk `whole` left of the diagonal
    if (lead) {
      uint4* ch = reinterpret_cast<uint4*>(row + ((whole ^ (r & 7)) << 4));
      uint4 v = *ch;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (e < lead) w[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
      *ch = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <bool FUSED>
__global__ void __launch_bounds__(192, 1)
    hgemm_tri_leaves_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmL,
                               const __grid_constant__ CUtensorMap tmC, const TcArgs p,
                               const TriLeaves leaves, const TriLeafExt lext) {
  using Cfg = LeafCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + Cfg::OFF_A;
  const uint32_t sB = sbase + Cfg::OFF_B;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t drain_bar = bar0 + 8 * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // producer's arrive.expect_tx (+ TMA bytes)
      mbar_init(empty_bar(s), 1);  // MMA issuer's tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), Cfg::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmL);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // A, B and C may come from the previous launch on the stream
  grid_dependency_wait();
  grid_launch_dependents();

  // unit t: rows [128·mt, +128) of X with mt = t / leaves, for leaf t % leaves:
  // the CTAs at work share those rows of X (read from memory once) and the
  // leaves' operand rows, which stay in L2
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        const int mt = t / leaves.count, b = t - mt * leaves.count;
        const int off = static_cast<int>(leaves.off[b]);
        const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
        const int nke = lext.ext[b] / Cfg::BK;  // K blocks of the carried update
        for (int j = 0; j < nke + nkb; ++j) {
          // update blocks first (all nkb row boxes), then the triangle's,
          // widest first (kb + 1 row boxes)
          const int kb = j < nke ? nkb - 1 : nkb - 1 - (j - nke);
          const int x = j < nke ? off + nkb * Cfg::BK + j * Cfg::BK : off + kb * Cfg::BK;
          if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) {
            ok = false;
            break;
          }
          if (!(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
            mbar_arrive_expect_tx(full_bar(stage),
                                  static_cast<uint32_t>(Cfg::A_BYTES + (kb + 1) * Cfg::L_BOX_BYTES));
          tma_load_2d(sA + stage * Cfg::A_BYTES, &tmX, full_bar(stage), x, mt * Cfg::BM);
          for (int r = 0; r <= kb; ++r)
            tma_load_2d(sB + stage * Cfg::B_BYTES + r * Cfg::L_BOX_BYTES, &tmL, full_bar(stage), x,
                        off + r * Cfg::L_BOX_ROWS);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last min(issued, STAGES) loads land before the CTA exits.
      int s = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < issued && i < STAGES; ++i) {
        if (s == 0) {
          s = STAGES - 1;
          ph ^= 1u;
        } else {
          --s;
        }
        wait_drain(full_bar(s), ph, wd);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------- MMA warp: masks each stage, lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      const int b = t % leaves.count;
      const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
      const int nke = lext.ext[b] / Cfg::BK;
      int free_acc = 1;
      if (lane == 0) free_acc = wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, free_acc, 0)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      for (int j = 0; j < nke + nkb; ++j) {
        const bool update = j < nke;  // a K block of the carried update: whole rows, no mask
        const int kb = update ? nkb - 1 : nkb - 1 - (j - nke);
        // every lane waits for the copy: its masking stores come after it
        const int landed = wait_phase(full_bar(stage), phase, wd, kWdMmaFull) ? 1 : 0;
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        if (!update) mask_diagonal_block(smem + Cfg::OFF_B + stage * Cfg::B_BYTES + kb * Cfg::L_BOX_BYTES, lane);
        fence_proxy_async_smem();  // the tensor cores read the stage through the async proxy
        __syncwarp();
        if (lane == 0) {
          tc_fence_after_sync();
          const uint64_t a_desc = sdesc_kmajor_sw128(sA + stage * Cfg::A_BYTES);
          const uint64_t b_desc = sdesc_kmajor_sw128(sB + stage * Cfg::B_BYTES);
          const uint32_t idesc = idesc_f16_f32acc(Cfg::BM, (kb + 1) * Cfg::L_BOX_ROWS);
#pragma unroll
          for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
            mma_f16_ss(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty_bar(stage));  // frees the stage once read
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(accf_bar(acc));  // accumulator complete
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // Drain: every MMA issued above completes before TMEM is freed.
    if (lane == 0) {
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 = rows of this warp
    uint8_t* cbuf_base = smem + Cfg::OFF_C + q * Cfg::C_BUFS * Cfg::C_BOX_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cb = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const int mt = t / leaves.count, b = t - mt * leaves.count;
      const int off = static_cast<int>(leaves.off[b]);
      const int boxes = static_cast<int>(leaves.size[b]) / kEpiCols;
      int ok = 1;
      if (lane == 0) ok = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      const int y0 = mt * Cfg::BM + q * kEpiRows;
#pragma unroll 1
      for (int c = 0; c < boxes; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, v0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        if (c == boxes - 1) {
          // the whole accumulator has been read: hand it back to the MMA warp
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(acc));
        }
        if (y0 >= p.M) continue;  // rows past the end of X
        const int x0 = off + c * kEpiCols;
        if (lane == 0) bulk_wait_group_read<1>();  // the store two boxes ago has read this buffer
        __syncwarp();
        uint8_t* buf = cbuf_base + cb * Cfg::C_BOX_BYTES;
        stage_row64<FUSED>(buf + lane * 128, lane, v0, v1, p.epi, p.C, p.M, p.N, p.ldc,
                           static_cast<int64_t>(y0) + lane, x0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(buf), x0, y0);  // clipped at the last row of C
          bulk_commit_group();
        }
        cb ^= 1;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes finish with the grid
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Split-K leaves: with few units, the leaf that carries the most updates walks
// by far the most K blocks. Here one cluster of CL CTAs takes one unit (a
// 128-row tile of X, a whole leaf of s columns), each CTA a contiguous range
// of its K blocks: the carried update's blocks are shared out, and the last
// CTA also takes the triangle's blocks (widest first, so every CTA's first
// block initialises all s accumulator columns). The CL partial sums are then
// reduced through distributed shared memory, as in the split-K GEMM: the s
// columns are cut into CL ranges of whole 64-column boxes, the CTA of slice r
// owns range r; once an owner's own MMAs are done (its ring is free) it tells
// the slices that have a partial, each of them stages its 32 rows per warp of
// the owner's range in its own shared memory and pushes them with one bulk
// copy into the owner's ring, whose barrier counts the bytes; the owner adds
// the partials in slice order (the result does not depend on timing), applies
// alpha, rounds to FP16 and stores its range. A final cluster barrier keeps
// every CTA until the others are done, so no copy or remote arrival touches
// a CTA that has left (an owner reaches it only after its partials landed).
// A CTA with no K blocks (a leaf with few carried blocks) has no partial: it
// sends nothing and only owns.

// K blocks [j0, j1) of slice r out of cl, in the unit's block order (the nke
// carried blocks, then the nkb triangle blocks, which the last slice takes).
// A triangle block counts as 1.5 carried ones: it is narrower, but masked by
// the whole MMA warp (measured: the last slice of the longest leaf finished
// ~1.5 µs after the others with equal counts).
__device__ __forceinline__ void split_range(int nke, int nkb, int r, int cl, int& j0, int& j1) {
  const int per = (2 * nke + 3 * nkb + 2 * cl - 1) / (2 * cl);
  j0 = min(nke, r * per);
  j1 = r < cl - 1 ? min(nke, (r + 1) * per) : nke + nkb;
}

// Row grow of C, columns x0 .. x0+63 (v0: the first 32, v1: the rest),
// rounded to FP16 (through the fused epilogue when FUSED) and stored with
// 16-byte stores (x0, N and ldc are multiples of 8 here). Rows past M are
// skipped.
template <bool FUSED>
__device__ __forceinline__ void store_row64(const uint32_t (&v0)[32], const uint32_t (&v1)[32],
                                            const EpiArgs& e, uint16_t* C, int64_t M, int64_t N,
                                            int64_t ldc, int64_t grow, int64_t x0) {
  if (grow >= M) return;
  uint16_t* out = C + grow * ldc + x0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (x0 + 8 * j >= N) break;
    if (!HG_DBG_INDEX(x0 + 8 * j + 7, N) || !HG_DBG_ALIGN(out + 8 * j, 16)) break;
    const uint32_t* v = (j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4));
    uint4 pk;
    if constexpr (FUSED) {
      pk = epi_pack8(v, e, load_c_old8(e, C, M, N, ldc, grow, x0 + 8 * j), load_bias8(e, x0 + 8 * j, N));
    } else {
      pk.x = pack_half2(v[0], v[1]);
      pk.y = pack_half2(v[2], v[3]);
      pk.z = pack_half2(v[4], v[5]);
      pk.w = pack_half2(v[6], v[7]);
    }
    *reinterpret_cast<uint4*>(out + 8 * j) = pk;
  }
}

// First 64-column box of the range owned by slice r, for a leaf of `boxes`
// boxes.
__host__ __device__ constexpr int owned_box(int r, int cl, int boxes) { return (boxes * r) / cl; }

// Swizzled FP32 block of `cols` columns: row q occupies cols·4 bytes at
// q·cols·4, and its 16-byte chunk c sits at chunk position c ^ (q % 8), so the
// 32 rows a warp writes at once spread over all banks.
__device__ __forceinline__ uint32_t split_block_offset(int q, int c, int cols) {
  return static_cast<uint32_t>(q * cols * 4 + ((c ^ (q & 7)) << 4));
}

template <int CL, bool FUSED>
__global__ void __launch_bounds__(192, 1)
    hgemm_tri_leaves_split_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmL,
                                  const __grid_constant__ CUtensorMap tmC, const TcArgs p,
                                  const TriLeaves leaves, const TriLeafExt lext) {
  using Cfg = LeafCfg;
  constexpr int STAGES = Cfg::STAGES;
  static_assert(CL >= 2 && CL <= 4, "one 64-column box per owner at least, four ready barriers");
  static_assert(2 * (CL - 1) * Cfg::BM * (Cfg::MAX_S / CL) * 4 <= Cfg::OFF_C, "the exchange fits in the ring");
  static_assert(2 * STAGES + 3 + CL <= Cfg::NUM_BARS, "the barriers fit");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + Cfg::OFF_A;
  const uint32_t sB = sbase + Cfg::OFF_B;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t accf_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = accf_bar + 8u;
  const uint32_t recv_bar = drain_bar + 8u;
  const uint32_t ready_bar0 = recv_bar + 8u;   // ready_bar0 + 8o: owner o may receive
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (STAGES + st); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = static_cast<int>(cluster_ctarank());
  const int u = blockIdx.x / CL;
  const int mt = u / leaves.count, b = u - mt * leaves.count;
  const int off = static_cast<int>(leaves.off[b]);
  const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
  const int nke = lext.ext[b] / Cfg::BK;
  const int boxes = nkb;  // 64-column boxes of the leaf
  int j0, j1;
  split_range(nke, nkb, r, CL, j0, j1);
  auto has_partial = [&](int sl) {
    int a0, a1;
    split_range(nke, nkb, sl, CL, a0, a1);
    return a1 > a0;
  };
  auto own_box0 = [&](int sl) { return owned_box(sl, CL, boxes); };
  auto own_cols = [&](int sl) { return 64 * (owned_box(sl + 1, CL, boxes) - owned_box(sl, CL, boxes)); };
  const bool mine = j1 > j0;  // this CTA has a partial
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    // the other slices' partials of this CTA's range
    int senders = 0;
    for (int sl = 0; sl < CL; ++sl)
      if (sl != r && has_partial(sl)) ++senders;
    mbar_init(recv_bar, 1);
    mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(senders * Cfg::BM * own_cols(r) * 4));
    for (int o = 0; o < CL; ++o) mbar_init(ready_bar0 + 8u * o, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmL);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::ACC_COLS);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();  // the TMEM address and the abort flag, within the CTA
  cluster_sync_after_init();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // A, B and C may come from the previous launch on the stream
  grid_dependency_wait();
  grid_launch_dependents();

  int ok = 1;
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int j = j0; j < j1; ++j) {
        // carried blocks: all nkb row boxes; triangle blocks: kb + 1 of them
        const int kb = j < nke ? nkb - 1 : nkb - 1 - (j - nke);
        const int x = j < nke ? off + nkb * Cfg::BK + j * Cfg::BK : off + kb * Cfg::BK;
        if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) break;
        if (!(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
          mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(Cfg::A_BYTES + (kb + 1) * Cfg::L_BOX_BYTES));
        tma_load_2d(sA + stage * Cfg::A_BYTES, &tmX, full_bar(stage), x, mt * Cfg::BM);
        for (int rb = 0; rb <= kb; ++rb)
          tma_load_2d(sB + stage * Cfg::B_BYTES + rb * Cfg::L_BOX_BYTES, &tmL, full_bar(stage), x,
                      off + rb * Cfg::L_BOX_ROWS);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Drain: the last min(issued, STAGES) loads land before the ring is reused.
      int st = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < issued && i < STAGES; ++i) {
        if (st == 0) {
          st = STAGES - 1;
          ph ^= 1u;
        } else {
          --st;
        }
        wait_drain(full_bar(st), ph, wd);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------- MMA warp: masks each stage, lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    bool good = true;
    for (int j = j0; j < j1; ++j) {
      const bool update = j < nke;
      const int kb = update ? nkb - 1 : nkb - 1 - (j - nke);
      const int landed = wait_phase(full_bar(stage), phase, wd, kWdMmaFull) ? 1 : 0;
      if (!__all_sync(0xffffffffu, landed)) {
        good = false;
        break;
      }
      if (!update) {
        mask_diagonal_block(smem + Cfg::OFF_B + stage * Cfg::B_BYTES + kb * Cfg::L_BOX_BYTES, lane);
        fence_proxy_async_smem();  // the tensor cores read the masked stage through the async proxy
      }
      __syncwarp();
      if (lane == 0) {
        tc_fence_after_sync();
        const uint64_t a_desc = sdesc_kmajor_sw128(sA + stage * Cfg::A_BYTES);
        const uint64_t b_desc = sdesc_kmajor_sw128(sB + stage * Cfg::B_BYTES);
        const uint32_t idesc = idesc_f16_f32acc(Cfg::BM, (kb + 1) * Cfg::L_BOX_ROWS);
#pragma unroll
        for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
          mma_f16_ss(tmem_base, a_desc + 2u * k, b_desc + 2u * k, idesc, (j > j0 || k > 0) ? 1u : 0u);
        mma_commit(empty_bar(stage));
      }
      __syncwarp();
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (lane == 0) {
      if (good && mine) mma_commit(accf_bar);  // the partial is complete
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // epilogue warps: the partial is complete, and the operand ring is free
    if (mine) {
      if (lane == 0) ok = wait_phase(accf_bar, 0, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    tc_fence_after_sync();
    // tell the slices that have a partial that they may send theirs of this
    // CTA's range (relaxed: the ring's last readers, the MMAs, completed
    // before accf did; a CTA without a partial never used its ring)
    if (warp == 2 && lane == 0 && ok && own_cols(r) > 0)
      for (int sl = 0; sl < CL; ++sl)
        if (sl != r && has_partial(sl))
          mbar_arrive_cluster_relaxed(mapa_shared(ready_bar0 + 8u * r, static_cast<uint32_t>(sl)));
  }

  const int q = warp & 3;  // TMEM lanes / tile rows 32q .. 32q+31
  const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const int row = q * 32 + lane;
  const int oc = own_cols(r);
  const int ox0 = 64 * own_box0(r);  // first column of the owned range, within the leaf
  // ring layout for the exchange: receive slots (one per other slice), then
  // the send staging
  const uint32_t recv_base = sbase;
  const uint32_t send_base = sbase + static_cast<uint32_t>((CL - 1) * Cfg::BM * (64 * ((boxes + CL - 1) / CL)) * 4);
  if (warp >= 2 && ok) {
    if (mine) {
      // every other owner's range of this warp's 32 rows, into the send
      // staging (this CTA's own ring) ...
      uint32_t send_off = send_base;
      for (int o = 0; o < CL; ++o) {
        const int cols = own_cols(o);
        if (o == r || cols == 0) continue;
        const int c0 = 64 * own_box0(o);
        uint8_t* blk = smem + (send_off - sbase);
#pragma unroll 1
        for (int c32 = 0; c32 < cols / 32; ++c32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + c0 + c32 * 32, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int w = 0; w < 8; ++w)
            *reinterpret_cast<uint4*>(blk + split_block_offset(row, c32 * 8 + w, cols)) =
                make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
        }
        send_off += static_cast<uint32_t>(Cfg::BM * cols * 4);
      }
      fence_proxy_async_smem();
      __syncwarp();
      // ... then one bulk copy per owner once its ring is free
      send_off = send_base;
      for (int o = 0; o < CL; ++o) {
        const int cols = own_cols(o);
        if (o == r || cols == 0) continue;
        int rdy = 1;
        if (lane == 0) rdy = wait_phase_cluster(ready_bar0 + 8u * o, 0, wd, kWdReduce) ? 1 : 0;
        rdy = __shfl_sync(0xffffffffu, rdy, 0);
        if (!rdy) {
          ok = 0;
          break;
        }
        if (lane == 0) {
          // this warp's 32 rows, into owner o's slot for slice r
          const int idx = r < o ? r : r - 1;
          const uint32_t rows_off = static_cast<uint32_t>(q * 32 * cols * 4);
          const uint32_t dst = mapa_shared(recv_base + idx * Cfg::BM * cols * 4 + rows_off, static_cast<uint32_t>(o));
          bulk_copy_to_cluster(dst, send_off + rows_off, static_cast<uint32_t>(32 * cols * 4),
                               mapa_shared(recv_bar, static_cast<uint32_t>(o)));
        }
        send_off += static_cast<uint32_t>(Cfg::BM * cols * 4);
      }
    }
    if (ok && oc > 0) {
      // own range: wait for the other slices' partials, add in slice order
      int got = 1;
      if (lane == 0) got = wait_phase_cluster(recv_bar, 0, wd, kWdReduce) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (got) {
        const int x0 = off + ox0;
        const int y0 = mt * Cfg::BM + q * kEpiRows;
        if constexpr (FUSED)
          prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc, static_cast<int64_t>(y0) + lane, x0, oc);
#pragma unroll 1
        for (int c64 = 0; c64 < oc / 64; ++c64) {
          float acc[64];
          bool first = true;
          for (int sl = 0; sl < CL; ++sl) {
            if (!has_partial(sl)) continue;
            if (sl == r) {
              uint32_t v0[32], v1[32];
              tmem_ld_32x32b_x32(t_row + ox0 + c64 * 64, v0);
              tmem_ld_32x32b_x32(t_row + ox0 + c64 * 64 + 32, v1);
              tmem_ld_wait(v0);
              tmem_ld_wait(v1);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                acc[i] = first ? __uint_as_float(v0[i]) : acc[i] + __uint_as_float(v0[i]);
                acc[32 + i] = first ? __uint_as_float(v1[i]) : acc[32 + i] + __uint_as_float(v1[i]);
              }
            } else {
              const int idx = sl < r ? sl : sl - 1;
              const uint8_t* blk = smem + idx * Cfg::BM * oc * 4;
#pragma unroll
              for (int w = 0; w < 16; ++w) {
                const float4 f = *reinterpret_cast<const float4*>(blk + split_block_offset(row, c64 * 16 + w, oc));
                acc[4 * w] = first ? f.x : acc[4 * w] + f.x;
                acc[4 * w + 1] = first ? f.y : acc[4 * w + 1] + f.y;
                acc[4 * w + 2] = first ? f.z : acc[4 * w + 2] + f.z;
                acc[4 * w + 3] = first ? f.w : acc[4 * w + 3] + f.w;
              }
            }
            first = false;
          }
          uint32_t v0[32], v1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] = __float_as_uint(acc[i]);
            v1[i] = __float_as_uint(acc[32 + i]);
          }
          // one row of 64 columns per thread, straight from registers
          store_row64<FUSED>(v0, v1, p.epi, const_cast<uint16_t*>(p.C), p.M, p.N, p.ldc,
                             static_cast<int64_t>(y0) + lane, x0 + c64 * 64);
        }
      } else {
        ok = 0;
      }
    }
  }

  // Leaving: an owner arrives here only after its partials have landed, so
  // once every CTA of the cluster has arrived no copy reads or writes a
  // CTA's shared memory and no remote arrival is pending.
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::ACC_COLS);
  cluster_sync();
}

// Clusters of CL CTAs of the split kernel that the device holds at once (0:
// none, e.g. on a partition too small for them), measured once per device.
template <int CL>
int split_clusters_resident(int dev, int sms) {
  static std::atomic<int> cached[64];  // count + 1; 0: not measured
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev] - 1;
  auto kern = hgemm_tri_leaves_split_kernel<CL, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LeafCfg::SMEM_BYTES) == cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((sms / CL) * CL));
    cfg.blockDim = dim3(LeafCfg::THREADS);
    cfg.dynamicSmemBytes = LeafCfg::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (dev >= 0 && dev < 64) cached[dev] = n + 1;
  return n;
}

}  // namespace

cudaError_t launch_tri_leaves_tc(const CUtensorMap& x, const CUtensorMap& l, const CUtensorMap& c,
                                 const TcArgs& args, const TriLeaves& leaves, const TriLeafExt& ext,
                                 cudaStream_t stream) {
  static std::atomic<bool> attr_done[3][2][64];
  const int fused = args.epi.mode != 0 ? 1 : 0;
  for (int b = 0; b < leaves.count; ++b)
    if (leaves.size[b] <= 0 || leaves.size[b] > LeafCfg::MAX_S || leaves.size[b] % LeafCfg::BK != 0 ||
        ext.ext[b] < 0 || ext.ext[b] % LeafCfg::BK != 0)
      return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // Few units (a short X): each unit's K blocks split over a cluster of four
  // CTAs when four times the units fit in one wave, else of two when twice
  // the units do, and when the device holds that many such clusters at once.
  const int64_t units = args.num_tiles;
  const int slices = units * 4 <= sms && units <= split_clusters_resident<4>(dev, sms)   ? 4
                     : units * 2 <= sms && units <= split_clusters_resident<2>(dev, sms) ? 2
                                                                                         : 1;
  auto kern = slices == 4 ? (fused ? hgemm_tri_leaves_split_kernel<4, true> : hgemm_tri_leaves_split_kernel<4, false>)
              : slices == 2 ? (fused ? hgemm_tri_leaves_split_kernel<2, true> : hgemm_tri_leaves_split_kernel<2, false>)
                            : (fused ? hgemm_tri_leaves_tc_kernel<true> : hgemm_tri_leaves_tc_kernel<false>);
  const int kind = slices == 4 ? 2 : slices == 2 ? 1 : 0;
  if (dev < 0 || dev >= 64 || !attr_done[kind][fused][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LeafCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[kind][fused][dev] = true;
  }
  if (slices > 1) {
    PdlLaunch pl(dim3(static_cast<unsigned>(units * slices)), dim3(LeafCfg::THREADS), LeafCfg::SMEM_BYTES, stream);
    pl.cluster(static_cast<unsigned>(slices));
    return cudaLaunchKernelEx(&pl.cfg, kern, x, l, c, args, leaves, ext);
  }
  PdlLaunch pl(dim3(static_cast<unsigned>(args.grid)), dim3(LeafCfg::THREADS), LeafCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&pl.cfg, kern, x, l, c, args, leaves, ext);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(trileaf)

}  // namespace hg
