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
//   * with few units (a short X: m of a few hundred rows), each leaf is cut
//     into 64-column parts (p.part_cols = 64), one unit each: part q takes
//     rows 64q .. 64q+63 of L_b (N = 64), the carried update's K blocks and
//     the triangle's K blocks kb ≥ q (the blocks below are zero for those
//     rows), masking block q. Four times as many SMs then share the longest
//     leaves' operand streams, each reading the X tile and a quarter of the
//     triangle rows;
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
  // With 64-column parts a stage needs only the X tile and one row box
  // (24 KB): the same ring space then holds twice the stages, interleaved.
  static constexpr int PART_STAGE_BYTES = A_BYTES + L_BOX_BYTES;
  static constexpr int PART_STAGES = STAGES * (A_BYTES + B_BYTES) / PART_STAGE_BYTES;  // 8
  static constexpr int MAX_STAGES = PART_STAGES;
  static constexpr int NUM_BARS = 2 * MAX_STAGES + 4 + 1;      // full, empty, acc full/empty, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;      // tmem address, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;      // + slack to align the base
  static constexpr int THREADS = 192;

  static_assert(PART_STAGES * PART_STAGE_BYTES <= STAGES * (A_BYTES + B_BYTES) && PART_STAGES >= STAGES,
                "the parts' stages fit in the ring");
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
  constexpr int MAXST = Cfg::MAX_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + Cfg::OFF_A;
  const uint32_t sB = sbase + Cfg::OFF_B;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t drain_bar = bar0 + 8 * (2 * MAXST + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (MAXST + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * MAXST + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * MAXST + 2 + b); };
  // the ring: Cfg::STAGES stages of an X tile and up to four row boxes
  // (whole leaves), or Cfg::PART_STAGES of an X tile and one row box (parts)
  const int parts = p.part_cols > 0 ? Cfg::MAX_S / p.part_cols : 1;
  const int nstages = parts > 1 ? Cfg::PART_STAGES : Cfg::STAGES;
  auto stage_a = [&](int s) {
    return parts > 1 ? sA + s * Cfg::PART_STAGE_BYTES : sA + s * Cfg::A_BYTES;
  };
  auto stage_b = [&](int s) {
    return parts > 1 ? sA + s * Cfg::PART_STAGE_BYTES + Cfg::A_BYTES : sB + s * Cfg::B_BYTES;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < MAXST; ++s) {
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
  // leaves' operand rows, which stay in L2. With parts (X then fits in L2),
  // leaf-major instead, so that the CTAs take the longest leaves' parts of
  // every tile first: u = t / parts = b·num_m + mt, part t % parts. A part
  // past a narrower leaf's columns is skipped by every role.
  auto decode = [&](int t, int& mt, int& b, int& part) {
    if (parts > 1) {
      const int u = t / parts;
      part = t - u * parts;
      b = u / p.num_m;
      mt = u - b * p.num_m;
    } else {
      part = 0;
      mt = t / leaves.count;
      b = t - mt * leaves.count;
    }
  };
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mt, b, part;
        decode(t, mt, b, part);
        const int off = static_cast<int>(leaves.off[b]);
        const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
        const int nke = lext.ext[b] / Cfg::BK;  // K blocks of the carried update
        if (parts > 1 && part >= nkb) continue;
        // triangle blocks: all of them (whole leaf), or kb ≥ part (a part)
        const int ntri = parts > 1 ? nkb - part : nkb;
        for (int j = 0; j < nke + ntri; ++j) {
          // update blocks first (all nkb row boxes), then the triangle's,
          // widest first (kb + 1 row boxes); a part loads its one row box
          const int kb = j < nke ? nkb - 1 : nkb - 1 - (j - nke);
          const int x = j < nke ? off + nkb * Cfg::BK + j * Cfg::BK : off + kb * Cfg::BK;
          const int r0 = parts > 1 ? part : 0, r1 = parts > 1 ? part : kb;
          if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) {
            ok = false;
            break;
          }
          if (!(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
            mbar_arrive_expect_tx(full_bar(stage),
                                  static_cast<uint32_t>(Cfg::A_BYTES + (r1 - r0 + 1) * Cfg::L_BOX_BYTES));
          tma_load_2d(stage_a(stage), &tmX, full_bar(stage), x, mt * Cfg::BM);
          for (int r = r0; r <= r1; ++r)
            tma_load_2d(stage_b(stage) + (r - r0) * Cfg::L_BOX_BYTES, &tmL, full_bar(stage), x,
                        off + r * Cfg::L_BOX_ROWS);
          ++issued;
          if (++stage == nstages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last min(issued, nstages) loads land before the CTA exits.
      int s = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < issued && i < nstages; ++i) {
        if (s == 0) {
          s = nstages - 1;
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
      int mt, b, part;
      decode(t, mt, b, part);
      const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
      const int nke = lext.ext[b] / Cfg::BK;
      if (parts > 1 && part >= nkb) continue;
      const int ntri = parts > 1 ? nkb - part : nkb;
      int free_acc = 1;
      if (lane == 0) free_acc = wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, free_acc, 0)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      for (int j = 0; j < nke + ntri; ++j) {
        const bool update = j < nke;  // a K block of the carried update: whole rows, no mask
        const int kb = update ? nkb - 1 : nkb - 1 - (j - nke);
        // every lane waits for the copy: its masking stores come after it
        const int landed = wait_phase(full_bar(stage), phase, wd, kWdMmaFull) ? 1 : 0;
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        // the diagonal sub-block: row box kb of the whole leaf, or the part's
        // own box when kb is the part's index (its other blocks are whole)
        if (!update && (parts == 1 || kb == part)) {
          mask_diagonal_block(smem + (stage_b(stage) - sbase) + (parts > 1 ? 0 : kb) * Cfg::L_BOX_BYTES, lane);
          fence_proxy_async_smem();  // the tensor cores read the masked stage through the async proxy
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after_sync();
          const uint64_t a_desc = sdesc_kmajor_sw128(stage_a(stage));
          const uint64_t b_desc = sdesc_kmajor_sw128(stage_b(stage));
          const uint32_t idesc = idesc_f16_f32acc(Cfg::BM, parts > 1 ? Cfg::L_BOX_ROWS : (kb + 1) * Cfg::L_BOX_ROWS);
#pragma unroll
          for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
            mma_f16_ss(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty_bar(stage));  // frees the stage once read
        }
        __syncwarp();
        if (++stage == nstages) {
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
      int mt, b, part;
      decode(t, mt, b, part);
      const int nkb = static_cast<int>(leaves.size[b]) / Cfg::BK;
      if (parts > 1 && part >= nkb) continue;
      // the part's one 64-column box, or the whole leaf's
      const int off = static_cast<int>(leaves.off[b]) + (parts > 1 ? part * kEpiCols : 0);
      const int boxes = parts > 1 ? 1 : static_cast<int>(leaves.size[b]) / kEpiCols;
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

}  // namespace

cudaError_t launch_tri_leaves_tc(const CUtensorMap& x, const CUtensorMap& l, const CUtensorMap& c,
                                 const TcArgs& args, const TriLeaves& leaves, const TriLeafExt& ext,
                                 cudaStream_t stream) {
  static std::atomic<bool> attr_done[2][64];
  const int fused = args.epi.mode != 0 ? 1 : 0;
  auto kern = fused ? hgemm_tri_leaves_tc_kernel<true> : hgemm_tri_leaves_tc_kernel<false>;
  for (int b = 0; b < leaves.count; ++b)
    if (leaves.size[b] <= 0 || leaves.size[b] > LeafCfg::MAX_S || leaves.size[b] % LeafCfg::BK != 0 ||
        ext.ext[b] < 0 || ext.ext[b] % LeafCfg::BK != 0)
      return cudaErrorInvalidValue;
  if (args.part_cols != 0 && args.part_cols != LeafCfg::L_BOX_ROWS) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[fused][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LeafCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[fused][dev] = true;
  }
  PdlLaunch pl(dim3(static_cast<unsigned>(args.grid)), dim3(LeafCfg::THREADS), LeafCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&pl.cfg, kern, x, l, c, args, leaves, ext);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(trileaf)

}  // namespace hg
