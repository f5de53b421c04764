// hgemm_tc2w.cu — the wide CTA-pair path of C = A·B on sm_103a: 256×512
// output tiles per pair of CTAs.
//
// Same contract as the other tensor-core paths (the HGEMM of "Nvidia Tensor
// Core-MMA PTX编程入门", §4 示例; FP32 accumulation per "GPU架构与CUDA",
// 混合精度核函数; zero-filled edges and clipped stores per "GPU架构与CUDA",
// 共享内存与分块).
//
// Why wider tiles: at 256×256 per pair the main loop is limited by the
// aggregate bandwidth from L2 to the SMs, not by the tensor cores (each SM
// needs 32 KB of operands per 64-wide K block for 2·128·256·64 flops). With
// 512 columns per pair, each SM loads 128 rows of A and 256 rows of B per K
// block (48 KB) for twice the MMA work: 25% fewer operand bytes per flop,
// without giving up any SM (clusters stay at two CTAs).
//
// Layout of the work:
//   * CTA r of a pair loads A rows [128r, 128r+128) of the tile and, for each
//     256-column half h of the tile, B rows [256h + 128r, 256h + 128r + 128)
//     (B stored N×K), into a 4-deep ring of 48 KB stages;
//   * the even CTA issues, per K step, two tcgen05.mma.cta_group::2 (M=256,
//     N=256, K=16), one per column half, into two FP32 accumulators that
//     together fill TMEM (2×256 columns);
//   * eight epilogue warps drain the two halves at once (warps 2..5 half 0,
//     warps 6..9 half 1, one TMEM lane quadrant each) and release each half
//     as soon as it is read; the next tile's MMAs for a half start then. The
//     whole 512-column accumulator fills TMEM, so this drain is the only
//     pause of the tensor cores between tiles, and two warps per quadrant
//     halve it (measured: +0.5% at 8192³, +1.6% at 4096³);
//   * serpentine K, epilogue, edges and watchdog as in hgemm_tc2.cu.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

struct WideCfg {
  static constexpr int BM = 2 * kTcBM;    // tile rows
  static constexpr int BN = 2 * kPairBN;  // tile columns (two 256-column halves)
  static constexpr int ROWS = kTcBM;      // A rows per CTA
  static constexpr int BROWS = kPairBN / 2;  // B rows per CTA per half
  static constexpr int BK = kTcBK;
  static constexpr int STAGES = 4;
  static constexpr int UMMA_K = 16;
  static constexpr int A_BYTES = ROWS * BK * 2;          // 16 KB
  static constexpr int BH_BYTES = BROWS * BK * 2;        // 16 KB per half
  static constexpr int B_BYTES = 2 * BH_BYTES;           // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB landed in each CTA
  static constexpr int TX_BYTES = 2 * STAGE_BYTES;        // expected by the even CTA
  static constexpr int EPI_WARPS = 8;  // four per column half
  static constexpr int C_BOX_BYTES = kEpiRows * kEpiCols * 2;
  static constexpr int C_BUFS = 1;
  static constexpr int C_BYTES = EPI_WARPS * C_BUFS * C_BOX_BYTES;
  static constexpr int HALF_COLS = kPairBN;              // TMEM columns per half
  static constexpr int TMEM_COLS = 2 * HALF_COLS;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_C + C_BYTES;
  // full[S], empty[S], accumulator full, accumulator-half empty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 1 + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, kPairBN);

  static_assert(A_BYTES % 1024 == 0 && BH_BYTES % 1024 == 0, "1024-byte aligned stages");
  static_assert(TMEM_COLS == 512, "two 256-column FP32 accumulators fill TMEM");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
};

// MN: the instantiation that also reads M-contiguous A or N-contiguous B
// (p.a_mn, p.b_mn) as MN-major tiles; the other one takes K-major operands.
template <bool FUSED, bool MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    hgemm_tc2w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const TcArgs p) {
  using Cfg = WideCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + Cfg::OFF_A;
  const uint32_t sB = sbase + Cfg::OFF_B;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t accf_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto acce_bar = [&](int h) { return bar0 + 8u * (2 * STAGES + 1 + h); };

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
    mbar_init(accf_bar, 1);                          // multicast tcgen05.commit per tile
    mbar_init(acce_bar(0), Cfg::EPI_WARPS);          // the pair's four warps of each half
    mbar_init(acce_bar(1), Cfg::EPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_cg2(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_alloc_permit_cg2();
  }
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
        int mb, nb;
        tile_coords(t, p.num_m, p.num_n, p.group_m, mb, nb);
        const int ya = mb * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS;
        const int yb = nb * Cfg::BN + static_cast<int>(rank) * Cfg::BROWS;
        // serpentine K (see hgemm_tc2.cu)
        const bool reverse = (((t - cluster_id) / num_clusters) & 1) != 0;
        for (int step = 0; step < p.num_kb; ++step) {
          const int kb = reverse ? p.num_kb - 1 - step : step;
          if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (rank == 0 && !(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
            mbar_arrive_expect_tx(full_bar(stage), Cfg::TX_BYTES);
          const uint32_t sb = sB + stage * Cfg::B_BYTES;
          if (MN && p.a_mn) {
            // A stored K×M: the CTA's 128 rows as two 64-row boxes, 8 KB apart
            tma_load_2d_cg2(sA + stage * Cfg::A_BYTES, &tmA, fb, ya, kb * Cfg::BK);
            tma_load_2d_cg2(sA + stage * Cfg::A_BYTES + kMnBoxBytes, &tmA, fb, ya + kMnBox, kb * Cfg::BK);
          } else {
            tma_load_2d_cg2(sA + stage * Cfg::A_BYTES, &tmA, fb, kb * Cfg::BK, ya);
          }
          if (MN && p.b_mn) {
            // B stored K×N: each half's 128 columns as two 64-column boxes
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_2d_cg2(sb + h * Cfg::BH_BYTES, &tmB, fb, yb + h * kPairBN, kb * Cfg::BK);
              tma_load_2d_cg2(sb + h * Cfg::BH_BYTES + kMnBoxBytes, &tmB, fb, yb + h * kPairBN + kMnBox,
                              kb * Cfg::BK);
            }
          } else {
            tma_load_2d_cg2(sb, &tmB, fb, kb * Cfg::BK, yb);
            tma_load_2d_cg2(sb + Cfg::BH_BYTES, &tmB, fb, kb * Cfg::BK, yb + kPairBN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain, as in the 256×256 pair kernel.
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
      uint32_t tile_phase = 0;  // parity of this CTA's tile count
      bool ok = true;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        for (int kb = 0; ok && kb < p.num_kb; ++kb) {
          if (!wait_phase(full_bar(stage), phase, wd, kWdMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // K-major: 16 K elements are 32 bytes along the row; MN-major: 16 K
          // rows of 128 bytes
          const bool a_mn = MN && p.a_mn, b_mn = MN && p.b_mn;
          const uint64_t a_desc = a_mn ? sdesc_mnmajor_sw128(sA + stage * Cfg::A_BYTES)
                                       : sdesc_kmajor_sw128(sA + stage * Cfg::A_BYTES);
          const uint32_t a_step = a_mn ? 128u : 2u, b_step = b_mn ? 128u : 2u;
          const uint32_t idesc = Cfg::IDESC | idesc_major_bits(a_mn, b_mn);
          const uint32_t sb = sB + stage * Cfg::B_BYTES;
          for (int h = 0; h < 2; ++h) {
            if (kb == 0) {
              // the previous tile's half h must have been drained
              if (!wait_phase_cluster(acce_bar(h), tile_phase ^ 1u, wd, kWdMmaAccEmpty)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
            const uint64_t b_desc = b_mn ? sdesc_mnmajor_sw128(sb + h * Cfg::BH_BYTES)
                                         : sdesc_kmajor_sw128(sb + h * Cfg::BH_BYTES);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(h * Cfg::HALF_COLS);
#pragma unroll
            for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
              // kb counts K steps in load order; the first one overwrites
              mma_f16_ss_cg2(d_tmem, a_desc + a_step * k, b_desc + b_step * k, idesc,
                             (kb > 0 || k > 0) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit_cg2_multicast(empty_bar(stage), 0x3);  // frees the stage in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_cg2_multicast(accf_bar, 0x3);  // both halves of both CTAs complete
        tile_phase ^= 1u;
      }
      mma_commit_cg2_multicast(drain_bar, 0x1);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    // warps 2..5 drain column half 0, warps 6..9 half 1, concurrently
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* buf = smem + Cfg::OFF_C + (warp - 2) * Cfg::C_BOX_BYTES;
    uint32_t tile_phase = 0;
    for (int t = cluster_id; t < p.num_tiles; t += num_clusters) {
      int mb, nb;
      tile_coords(t, p.num_m, p.num_n, p.group_m, mb, nb);
      if constexpr (FUSED)
        prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc,
                       static_cast<int64_t>(mb) * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS + q * kEpiRows + lane,
                       static_cast<int64_t>(nb) * Cfg::BN + h * kPairBN, kPairBN);
      int ok = 1;
      if (lane == 0) ok = wait_phase(accf_bar, tile_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const int y0 = mb * Cfg::BM + static_cast<int>(rank) * Cfg::ROWS + q * kEpiRows;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(h * Cfg::HALF_COLS);
      constexpr int chunks = kPairBN / kEpiCols;
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, v0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        if (c == chunks - 1 && t + num_clusters < p.num_tiles) {
          // half h has been read: the next tile's MMAs may overwrite it (after
          // this CTA's last tile nothing waits, and the cluster-scope release
          // is skipped)
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(h), 0));
        }
        const int x0 = nb * Cfg::BN + h * kPairBN + c * kEpiCols;
        if (x0 >= p.N || y0 >= p.M) continue;
        if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the box
        __syncwarp();
        uint8_t* row = buf + lane * 128;
        // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
        stage_row64<FUSED>(row, lane, v0, v1, p.epi, p.C, p.M, p.N, p.ldc, static_cast<int64_t>(y0) + lane, x0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(buf), x0, y0);
          bulk_commit_group();
        }
      }
      tile_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes finish with the grid
    __syncwarp();
  }

  // Neither CTA frees TMEM before the pair's last MMA and last TMEM read;
  // execution order is all this barrier needs (nothing between the two CTAs
  // is in flight by now), so its arrive is relaxed.
  tc_fence_before_sync();
  cluster_sync_relaxed();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_cg2(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace

int wide_max_clusters(int num_sms) {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaFuncSetAttribute(hgemm_tc2w_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           WideCfg::SMEM_BYTES) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
    cfg.blockDim = dim3(WideCfg::THREADS);
    cfg.dynamicSmemBytes = WideCfg::SMEM_BYTES;
    if (cudaOccupancyMaxActiveClusters(&n, hgemm_tc2w_kernel<false, false>, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = num_sms / 2;
  cached[dev] = n;
  return n;
}

cudaError_t launch_tc_wide(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const TcArgs& args, cudaStream_t stream) {
  static std::atomic<bool> attr_done[4][64];
  const int fused = args.epi.mode != 0 ? 1 : 0;
  const int mn = (args.a_mn || args.b_mn) ? 1 : 0;
  auto kern = mn ? (fused ? hgemm_tc2w_kernel<true, true> : hgemm_tc2w_kernel<false, true>)
                 : (fused ? hgemm_tc2w_kernel<true, false> : hgemm_tc2w_kernel<false, false>);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[2 * mn + fused][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WideCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[2 * mn + fused][dev] = true;
  }
  PdlLaunch l(dim3(static_cast<unsigned>(args.grid)), dim3(WideCfg::THREADS), WideCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, kern, a, b, c, args);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(tc2w)

}  // namespace hg
