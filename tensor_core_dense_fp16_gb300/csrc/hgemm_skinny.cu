// hgemm_skinny.cu — C = A·B when the output has too few 256×256 tiles to
// occupy the GPU (a small N or M against a long K, e.g. 4096×256×4096: the
// off-diagonal update of a recursive TRMM with a 4096×256 right-hand side, as
// in "异构计算中高性能TRMM与TRSM的递归算法实现", §2.2 and §5.1). Such shapes are
// bound by the bytes of A, so the design goal is that every SM streams A.
//
// Same contract as the other paths ("Nvidia Tensor Core-MMA PTX编程入门", §4
// 示例; FP32 accumulation, "GPU架构与CUDA", 混合精度核函数; zero-filled edges and
// clipped stores, "GPU架构与CUDA", 共享内存与分块).
//
// Design:
//   * one cluster of 2·S CTAs per 256×BN output tile (BN = 256 with S = 2, 3
//     or 4 slices, or BN = 128 with S = 2: half the partial sums to exchange
//     for the same operand bytes per SM); CTA rank r belongs to K-slice
//     p = r / 2 and tile half h = r % 2; pair p (ranks 2p, 2p+1) runs the
//     CTA-pair main loop of hgemm_tc2.cu over its contiguous range of 64-wide
//     K blocks, so A is read from memory exactly once over the grid;
//   * each CTA ends with a 128×BN FP32 partial sum in its TMEM;
//   * the S partials of a half are reduced through distributed shared
//     memory: the columns are cut into S ranges of whole 64-column units, the
//     CTA of slice p owns range p. Once an owner's own MMAs are done (its
//     operand ring is free) it tells the senders of its half; each sender's
//     epilogue warps stage their 32 rows of the owner's range in their own
//     shared memory and push them with one bulk copy into the owner's ring,
//     whose barrier counts the bytes. Each owner then adds the S partials in
//     slice order (so the result does not depend on timing), rounds to FP16
//     and TMA-stores its block of C, and acknowledges, so that no copy
//     touches a CTA that has left.
// No global scratch memory is used.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

// Column range of K-slice p: [64·owned_unit(p), 64·owned_unit(p + 1)), in
// 64-column units of a tile `units` units wide.
__host__ __device__ constexpr int owned_unit(int p, int split, int units) { return (units * p) / split; }

template <int SPLIT, int BN_>
struct SkCfg {
  static constexpr int BM = 2 * kTcBM;   // tile rows (both CTAs of a pair)
  static constexpr int BN = BN_;         // tile columns: 256 or 128
  static constexpr int UNITS = BN / 64;
  static constexpr int ROWS = kTcBM;     // rows per CTA
  static constexpr int BROWS = BN / 2;   // B rows per CTA
  static_assert(BROWS % kMnBox == 0, "an N-contiguous B arrives in whole 64-column boxes");
  static constexpr int BK = kTcBK;
  static constexpr int STAGES = BN == 256 ? 7 : 9;  // 32 KB or 24 KB per stage
  static constexpr int UMMA_K = 16;
  static constexpr int A_BYTES = ROWS * BK * 2;
  static constexpr int B_BYTES = BROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TX_BYTES = 2 * STAGE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;     // reused for the reduction and the C staging
  // the last slice owns the most units
  static constexpr int MAX_OWN_COLS = 64 * (owned_unit(SPLIT, SPLIT, UNITS) - owned_unit(SPLIT - 1, SPLIT, UNITS));
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int C_WARP_BYTES = kEpiRows * MAX_OWN_COLS * 2;
  static constexpr int C_BYTES = 4 * C_WARP_BYTES;
  // bytes a CTA owning `cols` columns receives (S-1 blocks) plus sends
  // (its partial outside its range), FP32, 128 rows; the most for the
  // largest range
  static constexpr int exchange_bytes(int cols) {
    return (SPLIT - 1) * ROWS * cols * 4 + ROWS * (BN - cols) * 4;
  }
  // The FP16 staging of C, inside the ring after the exchange area: the ring
  // is free once the CTA's own MMAs are done, and the staging is written only
  // after the received partials have been summed (so the ring holds one more
  // stage than with a separate staging area).
  static constexpr int OFF_C = (exchange_bytes(MAX_OWN_COLS) + 1023) / 1024 * 1024;
  static constexpr int RING_END = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = RING_END;
  // full, empty, accumulator full, drain, partials received, owner ready
  // (one per slice), partials acknowledged
  static constexpr int NUM_BARS = 2 * STAGES + 3 + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 192;
  static constexpr int TMEM_COLS = BN;
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);

  static_assert(OFF_C + C_BYTES <= RING_BYTES, "reduction and C staging fit in the ring");
  static_assert(exchange_bytes(64) <= RING_BYTES, "reduction fits in the ring");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(C_WARP_BYTES % 1024 == 0, "staging boxes stay 1024-byte aligned");
  static_assert(SPLIT <= UNITS, "every slice owns at least one 64-column unit");
};

// Swizzled FP32 block of `cols` columns: row r occupies cols*4 bytes at
// r*cols*4, and its 16-byte chunk c sits at chunk position c ^ (r % 8), so
// the 32 rows written by a warp at once spread over all banks.
__device__ __forceinline__ uint32_t f32_block_offset(int r, int c, int cols) {
  return static_cast<uint32_t>(r * cols * 4 + ((c ^ (r & 7)) << 4));
}

template <int SPLIT, int BN, bool FUSED>
__global__ void __launch_bounds__(192, 1)
    hgemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcArgs p) {
  using Cfg = SkCfg<SPLIT, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + Cfg::OFF_A;
  const uint32_t sB = sbase + Cfg::OFF_B;
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t accf_bar = bar0 + 8u * (2 * Cfg::STAGES);
  const uint32_t drain_bar = accf_bar + 8u;
  const uint32_t recv_bar = drain_bar + 8u;
  const uint32_t ready_bar0 = recv_bar + 8u;     // ready_bar0 + 8j: owner j may receive
  const uint32_t ack_bar = ready_bar0 + 8u * 4;  // every owner has received from us
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (Cfg::STAGES + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int slice = static_cast<int>(rank >> 1);  // K-slice p
  const int half = static_cast<int>(rank & 1);    // tile rows [128h, 128h+128)
  const uint32_t leader = rank & ~1u;             // even CTA of this pair
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << leader);
  const int tile = blockIdx.x / (2 * SPLIT);
  const int mb = tile / p.num_n;
  const int nb = tile % p.num_n;
  const int kb0 = static_cast<int>(static_cast<long long>(p.num_kb) * slice / SPLIT);
  const int kb1 = static_cast<int>(static_cast<long long>(p.num_kb) * (slice + 1) / SPLIT);
  const int own_c0 = 64 * owned_unit(slice, SPLIT, Cfg::UNITS);  // this CTA's column range
  const int own_cols = 64 * owned_unit(slice + 1, SPLIT, Cfg::UNITS) - own_c0;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(recv_bar, 1);
    // the partials of the other slices for this CTA's range, from 4 warps each
    mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((SPLIT - 1) * Cfg::ROWS * own_cols * 4));
    for (int j = 0; j < 4; ++j) mbar_init(ready_bar0 + 8u * j, 1);
    mbar_init(ack_bar, SPLIT - 1);
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

  int ok = 1;
  if (warp == 0) {
    // ------------------------------------------------ TMA producer (all CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      const int ya = mb * Cfg::BM + half * Cfg::ROWS;
      const int yb = nb * Cfg::BN + half * Cfg::BROWS;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) break;
        const uint32_t fb = mapa_shared(full_bar(stage), leader);
        if (rank == leader && !(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
          mbar_arrive_expect_tx(full_bar(stage), Cfg::TX_BYTES);
        if (p.a_mn) {
          // A stored K×M: the CTA's 128 rows as two 64-row boxes, 8 KB apart
          tma_load_2d_cg2(sA + stage * Cfg::A_BYTES, &tmA, fb, ya, kb * Cfg::BK);
          tma_load_2d_cg2(sA + stage * Cfg::A_BYTES + kMnBoxBytes, &tmA, fb, ya + kMnBox, kb * Cfg::BK);
        } else {
          tma_load_2d_cg2(sA + stage * Cfg::A_BYTES, &tmA, fb, kb * Cfg::BK, ya);
        }
        if (p.b_mn) {
          // B stored K×N: the CTA's BROWS columns as 64-column boxes, 8 KB apart
#pragma unroll
          for (int bx = 0; bx < Cfg::BROWS; bx += kMnBox)
            tma_load_2d_cg2(sB + stage * Cfg::B_BYTES + (bx / kMnBox) * kMnBoxBytes, &tmB, fb, yb + bx,
                            kb * Cfg::BK);
        } else {
          tma_load_2d_cg2(sB + stage * Cfg::B_BYTES, &tmB, fb, kb * Cfg::BK, yb);
        }
        ++issued;
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      int s = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < issued && i < Cfg::STAGES; ++i) {
        if (s == 0) {
          s = Cfg::STAGES - 1;
          ph ^= 1u;
        } else {
          --s;
        }
        if (rank == leader)
          wait_drain(full_bar(s), ph, wd);
        else
          wait_drain_cluster(empty_bar(s), ph, wd);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------------------------- MMA issuer (even CTAs)
    if (rank == leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool good = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_phase(full_bar(stage), phase, wd, kWdMmaFull)) {
          good = false;
          break;
        }
        tc_fence_after_sync();
        // K-major: 16 K elements are 32 bytes along the row; MN-major: 16 K
        // rows of 128 bytes
        const uint64_t a_desc = p.a_mn ? sdesc_mnmajor_sw128(sA + stage * Cfg::A_BYTES)
                                       : sdesc_kmajor_sw128(sA + stage * Cfg::A_BYTES);
        const uint64_t b_desc = p.b_mn ? sdesc_mnmajor_sw128(sB + stage * Cfg::B_BYTES)
                                       : sdesc_kmajor_sw128(sB + stage * Cfg::B_BYTES);
        const uint32_t a_step = p.a_mn ? 128u : 2u, b_step = p.b_mn ? 128u : 2u;
        const uint32_t idesc = Cfg::IDESC | idesc_major_bits(p.a_mn != 0, p.b_mn != 0);
#pragma unroll
        for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
          mma_f16_ss_cg2(tmem_base, a_desc + a_step * k, b_desc + b_step * k, idesc,
                         (kb > kb0 || k > 0) ? 1u : 0u);
        mma_commit_cg2_multicast(empty_bar(stage), pair_mask);
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (good) mma_commit_cg2_multicast(accf_bar, pair_mask);
      mma_commit_cg2_multicast(drain_bar, static_cast<uint16_t>(1u << leader));
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // epilogue warps: this CTA's partial is complete once the pair's MMAs are
    if (lane == 0) ok = wait_phase(accf_bar, 0, wd, kWdEpiAccFull) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    tc_fence_after_sync();
    // this CTA's operand ring is now free: tell the other slices of the same
    // half that they may send their partials of our column range (relaxed:
    // the ring's last readers, the MMAs, completed before accf did)
    if (warp == 2 && lane == 0 && ok)
      for (int s2 = 0; s2 < SPLIT; ++s2)
        if (s2 != slice)
          mbar_arrive_cluster_relaxed(mapa_shared(ready_bar0 + 8u * slice, static_cast<uint32_t>(2 * s2 + half)));
  }

  const int q = warp & 3;  // TMEM lanes / tile rows 32q .. 32q+31 of this CTA
  const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const int row = q * 32 + lane;
  if (FUSED && warp >= 2)
    prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc, static_cast<int64_t>(mb) * Cfg::BM + half * Cfg::ROWS + row,
                   static_cast<int64_t>(nb) * Cfg::BN + own_c0, own_cols);
  // ring layout for the exchange: receive slots first, then send staging
  const uint32_t recv_base = sbase;
  const uint32_t send_base = sbase + static_cast<uint32_t>((SPLIT - 1) * Cfg::ROWS * own_cols * 4);
  if (warp >= 2 && ok) {
    uint32_t send_off = send_base;
    for (int j = 0; j < SPLIT; ++j) {
      if (j == slice) continue;
      const int c0 = 64 * owned_unit(j, SPLIT, Cfg::UNITS);
      const int cols = 64 * owned_unit(j + 1, SPLIT, Cfg::UNITS) - c0;
      uint8_t* blk = smem + (send_off - sbase);
      // owner j's ring must be free before our copy lands in it
      int rdy = 1;
      if (lane == 0) rdy = wait_phase_cluster(ready_bar0 + 8u * j, 0, wd, kWdReduce) ? 1 : 0;
      rdy = __shfl_sync(0xffffffffu, rdy, 0);
      if (!rdy) break;
#pragma unroll 1
      for (int c32 = 0; c32 < cols / 32; ++c32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c0 + c32 * 32, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(blk + f32_block_offset(row, c32 * 8 + u, cols)) =
              make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // this warp's 32 rows, into slot `slice` (counted among j's senders)
        const uint32_t dst_rank = static_cast<uint32_t>(2 * j + half);
        const int idx = slice < j ? slice : slice - 1;
        const uint32_t rows_off = static_cast<uint32_t>(q * 32 * cols * 4);
        const uint32_t dst = mapa_shared(recv_base + idx * Cfg::ROWS * cols * 4 + rows_off, dst_rank);
        bulk_copy_to_cluster(dst, send_off + rows_off, static_cast<uint32_t>(32 * cols * 4),
                             mapa_shared(recv_bar, dst_rank));
      }
      send_off += static_cast<uint32_t>(Cfg::ROWS * cols * 4);
    }

    // own range: wait for the other slices' blocks, add in slice order
    int got = 1;
    if (lane == 0) got = wait_phase_cluster(recv_bar, 0, wd, kWdReduce) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    // every copy into us has completed (its bytes were counted): the senders
    // may leave (relaxed: this reports completion already observed)
    if (got && warp == 2 && lane == 0)
      for (int s2 = 0; s2 < SPLIT; ++s2)
        if (s2 != slice) mbar_arrive_cluster_relaxed(mapa_shared(ack_bar, static_cast<uint32_t>(2 * s2 + half)));
    if (got) {
      const int x0 = nb * Cfg::BN + own_c0;
      const int y0 = mb * Cfg::BM + half * Cfg::ROWS + q * kEpiRows;
      uint8_t* cbuf = smem + Cfg::OFF_C + q * Cfg::C_WARP_BYTES;
#pragma unroll 1
      for (int c32 = 0; c32 < own_cols / 32; ++c32) {
        uint32_t own[32];
        tmem_ld_32x32b_x32(t_row + own_c0 + c32 * 32, own);
        tmem_ld_wait(own);
        float acc[32];
        for (int sl = 0; sl < SPLIT; ++sl) {
          if (sl == slice) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              acc[i] = (sl == 0) ? __uint_as_float(own[i]) : acc[i] + __uint_as_float(own[i]);
          } else {
            const int idx = sl < slice ? sl : sl - 1;
            const uint8_t* blk = smem + idx * Cfg::ROWS * own_cols * 4;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 f =
                  *reinterpret_cast<const float4*>(blk + f32_block_offset(row, c32 * 8 + u, own_cols));
              if (sl == 0) {
                acc[4 * u] = f.x;
                acc[4 * u + 1] = f.y;
                acc[4 * u + 2] = f.z;
                acc[4 * u + 3] = f.w;
              } else {
                acc[4 * u] += f.x;
                acc[4 * u + 1] += f.y;
                acc[4 * u + 2] += f.z;
                acc[4 * u + 3] += f.w;
              }
            }
          }
        }
        // 32 FP16 columns (64 bytes) into the 128-byte-swizzled staging box
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 pk;
          if constexpr (!FUSED) {
            pk.x = pack_half2(__float_as_uint(acc[8 * u]), __float_as_uint(acc[8 * u + 1]));
            pk.y = pack_half2(__float_as_uint(acc[8 * u + 2]), __float_as_uint(acc[8 * u + 3]));
            pk.z = pack_half2(__float_as_uint(acc[8 * u + 4]), __float_as_uint(acc[8 * u + 5]));
            pk.w = pack_half2(__float_as_uint(acc[8 * u + 6]), __float_as_uint(acc[8 * u + 7]));
          } else {
            uint32_t vb[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) vb[i] = __float_as_uint(acc[8 * u + i]);
            const int64_t col0 = static_cast<int64_t>(x0) + c32 * 32 + 8 * u;
            pk = epi_pack8(vb, p.epi, load_c_old8(p.epi, p.C, p.M, p.N, p.ldc, y0 + lane, col0),
                           load_bias8(p.epi, col0, p.N));
          }
          const int chunk = c32 * 4 + u;  // 16-byte chunk within the row
          const int box = chunk >> 3;     // 64-column box
          const int cin = chunk & 7;
          *reinterpret_cast<uint4*>(cbuf + box * (kEpiRows * 128) + lane * 128 +
                                    ((cin ^ (lane & 7)) << 4)) = pk;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && y0 < p.M) {
        for (int box = 0; box < own_cols / kEpiCols; ++box) {
          const int x = x0 + box * kEpiCols;
          if (x < p.N) tma_store_2d(&tmC, smem_u32(cbuf + box * (kEpiRows * 128)), x, y0);
        }
        bulk_commit_group();
        bulk_wait_group_read<0>();  // shared memory read; the writes finish with the grid
      }
      __syncwarp();
    }
  }

  // Leaving: every owner acknowledges once all partials have landed in its
  // shared memory, so after our acknowledgements no copy reads our shared
  // memory and nobody writes into it. The pair's collective TMEM release is
  // reached by both CTAs only after both are done with TMEM.
  if (warp == 2 && lane == 0 && ok) wait_phase_cluster(ack_bar, 0, wd, kWdReduce);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_cg2(tmem_base, Cfg::TMEM_COLS);
}

template <int SPLIT, int BN>
cudaError_t launch_split(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                         const TcArgs& args, cudaStream_t stream) {
  using Cfg = SkCfg<SPLIT, BN>;
  static std::atomic<bool> attr_done[2][64];
  const int fused = args.epi.mode != 0 ? 1 : 0;
  auto kern = fused ? hgemm_skinny_kernel<SPLIT, BN, true> : hgemm_skinny_kernel<SPLIT, BN, false>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[fused][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[fused][dev] = true;
  }
  PdlLaunch l(dim3(static_cast<unsigned>(args.num_tiles * 2 * SPLIT)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES,
              stream);
  l.cluster(2 * SPLIT);
  return cudaLaunchKernelEx(&l.cfg, kern, a, b, c, args);
}

template <int SPLIT, int BN>
int max_clusters_split(int num_sms) {
  using Cfg = SkCfg<SPLIT, BN>;
  auto kern = hgemm_skinny_kernel<SPLIT, BN, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) ==
      cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * SPLIT;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((num_sms / (2 * SPLIT)) * 2 * SPLIT));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  return n;
}

}  // namespace

int skinny_max_clusters(int split, int tile_n, int num_sms) {
  if (tile_n == 128) return split == 2 ? max_clusters_split<2, 128>(num_sms) : 0;
  switch (split) {
    case 2:
      return max_clusters_split<2, 256>(num_sms);
    case 3:
      return max_clusters_split<3, 256>(num_sms);
    case 4:
      return max_clusters_split<4, 256>(num_sms);
    default:
      return 0;
  }
}

cudaError_t launch_skinny(int split, int tile_n, const CUtensorMap& a, const CUtensorMap& b,
                          const CUtensorMap& c, const TcArgs& args, cudaStream_t stream) {
  if (tile_n == 128) return split == 2 ? launch_split<2, 128>(a, b, c, args, stream) : cudaErrorInvalidValue;
  if (tile_n != 256) return cudaErrorInvalidValue;
  switch (split) {
    case 2:
      return launch_split<2, 256>(a, b, c, args, stream);
    case 3:
      return launch_split<3, 256>(a, b, c, args, stream);
    case 4:
      return launch_split<4, 256>(a, b, c, args, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(skinny)

}  // namespace hg
