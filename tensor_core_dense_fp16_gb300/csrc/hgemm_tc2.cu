// hgemm_tc2.cu — the CTA-pair tensor-core path of C = A·B on sm_103a.
//
// Same contract as hgemm_tc.cu (the HGEMM of "Nvidia Tensor Core-MMA
// PTX编程入门", §4 示例, FP32 accumulation per "GPU架构与CUDA", 混合精度核函数,
// zero-filled edges and clipped stores per "GPU架构与CUDA", 共享内存与分块), with
// a larger output tile shared by two SMs:
//   * clusters of two CTAs (one per SM of a TPC) own 256×256 output tiles;
//     CTA r of the pair loads rows [128r, 128r+128) of the tile's A slab and
//     rows [128r, 128r+128) of its B slab (B stored N×K), 64 K-columns per
//     stage, into a 6-deep ring of 128-byte-swizzled shared memory;
//   * the even CTA issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16): the
//     tensor cores of both SMs read both CTAs' operand halves, and each CTA's
//     TMEM receives its 128 accumulator rows (256 FP32 columns, two buffers);
//   * both CTAs' TMA loads complete on the even CTA's "full" barrier; MMA
//     completion is multicast to both CTAs' "empty" and "accumulator full"
//     barriers; both CTAs' epilogues release an accumulator buffer by arriving
//     on the even CTA's "accumulator empty" barrier;
//   * each CTA's four epilogue warps drain its TMEM half exactly as in the
//     single-CTA kernel (tcgen05.ld, round to nearest even, swizzled staging,
//     clipped TMA stores).
// Per SM, a stage is 32 KB instead of 48 KB for the same MMA work, which
// allows six stages in flight and halves each SM's share of B traffic. When
// every unit of a launch is a tile part, a stage shrinks to the part's bytes
// (24 or 20 KB) and the same ring holds eight or nine of them: an SM takes
// in at most ~112 GB/s, so more bytes in flight are what hides DRAM latency.
//
// Wave tail: when the tiles do not fill the last wave of clusters (or the
// only one), the tiles of that wave are cut into parts of 128 or 64 columns
// (N=128 or N=64 pair MMAs) so that two or four times as many clusters share
// them and the wave lasts a half or a quarter of a tile.
//
// Serpentine K: rounds of tiles alternate the direction in which they walk
// K, so each round starts on operand blocks that the previous round read
// last and that are still in L2 (measured: ~25% less DRAM traffic).
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

template <int MAX_STAGES_, int EPI_WARPS_ = 4>
struct PairCfg {
  static constexpr int BM = 2 * kTcBM;   // cluster tile rows
  static constexpr int BN = kPairBN;     // cluster tile columns
  static constexpr int ROWS = kTcBM;     // A rows per CTA
  static constexpr int BROWS = BN / 2;   // B rows (tile columns) per CTA
  static constexpr int BK = kTcBK;
  static constexpr int MAX_STAGES = MAX_STAGES_;
  static constexpr int UMMA_K = 16;
  static constexpr int A_BYTES = ROWS * BK * 2;
  static constexpr int B_BYTES = BROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // whole tiles: landed in each CTA
  static constexpr int TX_BYTES = 2 * STAGE_BYTES;          // expected by the even CTA
  static constexpr int RING_BYTES = kPairRingBytes;         // six whole-tile stages
  static_assert(RING_BYTES == 6 * STAGE_BYTES, "the ring holds six whole-tile stages");
  // plain products: four epilogue warps with two staging boxes each; fused
  // ones: eight (two per TMEM lane quarter, alternate 64-column boxes) with
  // one box each, since their epilogue arithmetic and reads of C take longer
  // than a short main loop
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "one or two epilogue warps per TMEM lane quarter");
  static constexpr int C_BOX_BYTES = kEpiRows * kEpiCols * 2;
  static constexpr int C_BUFS = EPI_WARPS == 8 ? 1 : 2;
  static constexpr int C_BYTES = EPI_WARPS * C_BUFS * C_BOX_BYTES;
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static constexpr int OFF_RING = 0;                        // stage s: A, then B
  static constexpr int OFF_C = OFF_RING + RING_BYTES;
  static constexpr int OFF_BAR = OFF_C + C_BYTES;
  static constexpr int NUM_BARS = 2 * MAX_STAGES + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);

  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte aligned stages");
  static_assert(RING_BYTES / (A_BYTES + 32 * BK * 2) <= MAX_STAGES, "barriers for the narrowest stages");
  static_assert(TMEM_COLS == 512, "two 256-column FP32 accumulators");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
};

// Work unit t: a whole 256×256 tile below p.full_tiles, else one part of
// p.part_cols (128 or 64) columns of a tile (256 / part_cols consecutive
// units per tile), in raster order. In a batched launch, whole tile w
// belongs to product w / p.batch_tiles, whose coordinates are shifted.
struct PairTile {
  int mb, nb;
  int n0;     // first column of C
  int ncols;  // 256, 128 or 64
  int koff;   // shift of the K coordinate of A and B
};

__device__ __forceinline__ PairTile pair_tile(int t, const TcArgs& p) {
  PairTile w;
  int whole = t, part = -1;
  if (t >= p.full_tiles) {
    const int parts = kPairBN / p.part_cols;
    const int h = t - p.full_tiles;
    whole = p.full_tiles + h / parts;
    part = h - (h / parts) * parts;
  }
  int shift = 0;
  if (p.batch_tiles > 0) {
    const int j = whole / p.batch_tiles;
    whole -= j * p.batch_tiles;
    shift = j * p.batch_shift;
  }
  tile_coords(whole, p.num_m, p.num_n, p.group_m, w.mb, w.nb);
  w.koff = shift;
  w.n0 = shift + w.nb * kPairBN + (part < 0 ? 0 : part * p.part_cols);
  w.ncols = part < 0 ? kPairBN : p.part_cols;
  return w;
}

template <int MAX_STAGES, bool FUSED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED ? 320 : 192, 1)
    hgemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmC,
                     const TcArgs p) {
  using Cfg = PairCfg<MAX_STAGES, FUSED ? 8 : 4>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  // ring geometry of this launch: p.stages stages of p.stage_bytes (A first)
  const int STAGES = p.stages;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.stage_bytes);
  const uint32_t sA = sbase + Cfg::OFF_RING;
  const uint32_t sB = sA + Cfg::A_BYTES;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t drain_bar = bar0 + 8 * (2 * MAX_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (MAX_STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * MAX_STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * MAX_STAGES + 2 + b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // even CTA's arrive.expect_tx; TMA bytes of both CTAs
      mbar_init(empty_bar(s), 1);  // multicast tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);                     // multicast tcgen05.commit
      mbar_init(acce_bar(b), 2 * Cfg::EPI_WARPS);    // every epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmBh);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_cg2(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_alloc_permit_cg2();
  }
  // barrier initialisation must be visible to the peer before any remote
  // arrive or TMA completion can target it
  tc_fence_before_sync();
  __syncthreads();  // the TMEM address and the abort flag, within the CTA
  cluster_sync_after_init();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // operands and C may come from the previous launch on the stream
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        const PairTile w = pair_tile(t, p);
        const bool whole = w.ncols == Cfg::BN;
        const int ya = w.mb * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS;
        const int yb = w.n0 + static_cast<int>(rank) * (w.ncols / 2);
        const CUtensorMap* mapb = whole ? &tmB : &tmBh;  // tmBh: part_cols / 2 rows per CTA
        const uint32_t tx = whole ? Cfg::TX_BYTES : 2u * (Cfg::A_BYTES + (w.ncols / 2) * Cfg::BK * 2);
        // serpentine K: every other round of tiles walks K backwards, so it
        // starts on the K blocks the previous round read last (still in L2)
        const bool reverse = (((t - cluster_id) / num_clusters) & 1) != 0;
        for (int step = 0; step < p.num_kb; ++step) {
          const int kb = reverse ? p.num_kb - 1 - step : step;
          if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const int kx = kb * Cfg::BK + w.koff;
          if (rank == 0 && !(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
            mbar_arrive_expect_tx(full_bar(stage), tx);
          if (p.a_mn) {
            // A stored K×M: the CTA's 128 rows as two 64-row boxes, 8 KB apart
            tma_load_2d_cg2(sA + stage * stage_bytes, &tmA, fb, ya, kx);
            tma_load_2d_cg2(sA + stage * stage_bytes + kMnBoxBytes, &tmA, fb, ya + kMnBox, kx);
          } else {
            tma_load_2d_cg2(sA + stage * stage_bytes, &tmA, fb, kx, ya);
          }
          if (p.b_mn) {
            // B stored K×N: the CTA's ncols/2 columns as 64-column boxes, 8 KB apart
            for (int bx = 0; bx < w.ncols / 2; bx += kMnBox)
              tma_load_2d_cg2(sB + stage * stage_bytes + (bx / kMnBox) * kMnBoxBytes, &tmB, fb, yb + bx, kx);
          } else {
            tma_load_2d_cg2(sB + stage * stage_bytes, mapb, fb, kx, yb);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain. The even CTA's full barriers count the bytes of both CTAs, so
      // their completion means both CTAs' copies landed. The odd CTA waits
      // instead until the MMAs consumed its last stages (the empty barrier
      // phase that follows each of its loads).
      int s = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < issued && i < STAGES; ++i) {
        if (s == 0) {
          s = STAGES - 1;
          ph ^= 1u;
        } else {
          --s;
        }
        if (rank == 0)
          wait_drain(full_bar(s), ph, wd);
        else
          wait_drain_cluster(empty_bar(s), ph, wd);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        const uint32_t idesc = (t < p.full_tiles ? Cfg::IDESC : idesc_f16_f32acc(Cfg::BM, p.part_cols)) |
                               idesc_major_bits(p.a_mn != 0, p.b_mn != 0);
        if (!wait_phase_cluster(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_phase(full_bar(stage), phase, wd, kWdMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // K-major: 16 K elements are 32 bytes along the row; MN-major: 16 K
          // rows of 128 bytes
          const uint64_t a_desc = p.a_mn ? sdesc_mnmajor_sw128(sA + stage * stage_bytes)
                                         : sdesc_kmajor_sw128(sA + stage * stage_bytes);
          const uint64_t b_desc = p.b_mn ? sdesc_mnmajor_sw128(sB + stage * stage_bytes)
                                         : sdesc_kmajor_sw128(sB + stage * stage_bytes);
          const uint32_t a_step = p.a_mn ? 128u : 2u, b_step = p.b_mn ? 128u : 2u;
#pragma unroll
          for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
            // kb counts the tile's K steps in load order (the producer may walk
            // K backwards); the first step overwrites the accumulator
            mma_f16_ss_cg2(d_tmem, a_desc + a_step * k, b_desc + b_step * k, idesc,
                           (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit_cg2_multicast(empty_bar(stage), 0x3);  // frees the stage in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_cg2_multicast(accf_bar(acc), 0x3);  // both TMEM halves complete
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit_cg2_multicast(drain_bar, 0x1);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else if constexpr (FUSED) {
    // --------------------------------------- fused epilogue (both CTAs)
    // warps 2..5 take the even 64-column boxes of a tile, warps 6..9 the odd
    // ones; warp w reads TMEM lanes 32·(w % 4) .. +31
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* buf = smem + Cfg::OFF_C + (warp - 2) * Cfg::C_BOX_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster_id; t < p.num_tiles; t += num_clusters) {
      const PairTile w = pair_tile(t, p);
      const int chunks = w.ncols / kEpiCols;
      const int64_t grow = static_cast<int64_t>(w.mb) * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS +
                           q * kEpiRows + lane;  // this lane's row of C
      prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc, grow, w.n0, w.ncols);
      int ok = 1;
      if (lane == 0) ok = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      const int y0 = w.mb * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS + q * kEpiRows;
      // this warp's last box (none when a 64-column part leaves the odd box out)
      const int last = (chunks - 1 - h) >= 0 ? h + ((chunks - 1 - h) / 2) * 2 : -1;
      // After a CTA's last tile no MMA waits for its accumulator again, so
      // its release (a cluster-scope release, ~1,000 cycles) is skipped.
      const bool reused = t + num_clusters < p.num_tiles;
      if (last < 0 && reused) {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
      }
#pragma unroll 1
      for (int c = h; c < chunks; c += 2) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, v0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        if (c == last && reused) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        const int x0 = w.n0 + c * kEpiCols;
        if (x0 >= p.N || y0 >= p.M) continue;
        if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the box
        __syncwarp();
        // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
        stage_row64<true>(buf + lane * 128, lane, v0, v1, p.epi, p.C, p.M, p.N, p.ldc, grow, x0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(buf), x0, y0);
          bulk_commit_group();
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes finish with the grid
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    uint8_t* cbuf_base = smem + Cfg::OFF_C + q * Cfg::C_BUFS * Cfg::C_BOX_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cb = 0;
    for (int t = cluster_id; t < p.num_tiles; t += num_clusters) {
      const PairTile w = pair_tile(t, p);
      const int chunks = w.ncols / kEpiCols;
      if constexpr (FUSED)
        prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc,
                       static_cast<int64_t>(w.mb) * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS + q * kEpiRows + lane,
                       w.n0, w.ncols);
      int ok = 1;
      if (lane == 0)
        ok = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      const int y0 = w.mb * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS + q * kEpiRows;
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, v0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        // no release after this CTA's last tile: no MMA waits for it again
        if (c == chunks - 1 && t + num_clusters < p.num_tiles) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        const int x0 = w.n0 + c * kEpiCols;
        if (x0 >= p.N || y0 >= p.M) continue;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* buf = cbuf_base + cb * Cfg::C_BOX_BYTES;
        uint8_t* row = buf + lane * 128;
        // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
        stage_row64<FUSED>(row, lane, v0, v1, p.epi, p.C, p.M, p.N, p.ldc, static_cast<int64_t>(y0) + lane, x0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(buf), x0, y0);
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

  // Neither CTA frees TMEM before the pair's last MMA and last TMEM read.
  // Execution order is all this barrier needs: no copy or remote arrival
  // between the two CTAs is in flight by now (the last tile's accumulator
  // is not released, the MMAs and loads completed on waited barriers), so
  // its arrive is relaxed (a release costs ~1,000 cycles).
  tc_fence_before_sync();
  cluster_sync_relaxed();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_cg2(tmem_base, Cfg::TMEM_COLS);
}

constexpr int kPairStages = 10;  // barriers for up to ten stages (the ring holds six to nine)

}  // namespace

int pair_max_clusters(int num_sms) {
  using Cfg = PairCfg<kPairStages>;
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  auto kern = hgemm_tc2_kernel<kPairStages, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = num_sms / 2;
  cached[dev] = n;
  return n;
}

int pair_smem_bytes() { return PairCfg<kPairStages>::SMEM_BYTES; }

cudaError_t launch_tc_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b_part,
                           const CUtensorMap& c, const TcArgs& args, cudaStream_t stream) {
  using Cfg = PairCfg<kPairStages, 4>;
  using FusedCfg = PairCfg<kPairStages, 8>;
  static_assert(Cfg::SMEM_BYTES == FusedCfg::SMEM_BYTES, "both instantiations have the same footprint");
  static std::atomic<bool> attr_done[2][64];
  const int fused = args.epi.mode != 0 ? 1 : 0;
  auto kern = fused ? hgemm_tc2_kernel<kPairStages, true> : hgemm_tc2_kernel<kPairStages, false>;
  const int threads = fused ? FusedCfg::THREADS : Cfg::THREADS;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[fused][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[fused][dev] = true;
  }
  PdlLaunch l(dim3(static_cast<unsigned>(args.grid)), dim3(static_cast<unsigned>(threads)), Cfg::SMEM_BYTES,
              stream);
  return cudaLaunchKernelEx(&l.cfg, kern, a, b, b_part, c, args);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(tc2)

}  // namespace hg
