// hgemm_tc.cu — the tensor-core path of C = A·B on sm_103a.
//
// What it computes: the HGEMM of "Nvidia Tensor Core-MMA PTX编程入门", §4 示例
// (A M×K row-major, B K×N column-major, C M×N row-major, FP16), with FP32
// accumulation as in "GPU架构与CUDA", 混合精度核函数, and the edge rule of
// "GPU架构与CUDA", 共享内存与分块 (out-of-range terms are zero, stores are
// clipped to C).
//
// How (a Blackwell design, not the page's warp-per-16×8-tile mma.sync kernel):
//   * persistent CTAs, one per SM, walk 128×256 output tiles in a grouped
//     raster order so that concurrently running tiles share A rows and B
//     columns in L2;
//   * warp 0 (one thread) streams 128×64 A and 256×64 B boxes with TMA into a
//     STAGES-deep ring of 128-byte-swizzled shared-memory buffers; both
//     operands are K-major, which is exactly the page's layout (A row-major,
//     B column-major), so no transpose is needed;
//   * warp 1 (one thread) issues tcgen05.mma (M=128, N=256, K=16) into an FP32
//     accumulator in tensor memory; TMEM holds two accumulators (2×256
//     columns) so the epilogue of one tile overlaps the main loop of the next;
//   * warps 2–5 read the accumulator with tcgen05.ld (each warp owns the 32
//     TMEM lanes = tile rows it may access), round to FP16 (round to nearest
//     even), stage 32×64 boxes in swizzled shared memory and write them with
//     TMA stores, which clip at the edges of C.
//   * Out-of-range rows, columns and K steps come back from TMA as zeros.
//   * Every mbarrier wait is bounded in time; a wait that gives up records a
//     code in the device watchdog word, raises a CTA-wide abort flag, and the
//     kernel drains its in-flight copies and MMAs, frees TMEM and returns.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {

__device__ int g_status_word = 0;

cudaError_t status_word_address(int** addr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(addr), g_status_word);
}

namespace {

template <int BN_, int STAGES_>
struct TcCfg {
  static constexpr int BM = kTcBM;
  static constexpr int BN = BN_;
  static constexpr int BK = kTcBK;
  static constexpr int STAGES = STAGES_;
  static constexpr int UMMA_K = 16;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS = 4;
  static constexpr int C_BOX_BYTES = kEpiRows * kEpiCols * 2;  // 4 KB
  static constexpr int C_BUFS = 2;                               // per epilogue warp
  static constexpr int C_BYTES = EPI_WARPS * C_BUFS * C_BOX_BYTES;
  static constexpr int ACC_COLS = BN;                            // FP32: one column per N
  static constexpr int TMEM_COLS = 2 * ACC_COLS;                 // double buffer
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_C + C_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;  // full, empty, acc full/empty, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem address, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base
  static constexpr int THREADS = 192;
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);

  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && C_BOX_BYTES % 1024 == 0,
                "swizzled buffers must stay 1024-byte aligned");
  static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 ||
                    TMEM_COLS == 512,
                "TMEM allocations are powers of two in [32, 512]");
  static_assert(BN % kEpiCols == 0 && BN >= 16 && BN <= 256 && BN % 16 == 0,
                "M=128 MMAs take N a multiple of 16 up to 256");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
};

template <int BN, int STAGES, bool FUSED>
__global__ void __launch_bounds__(192, 1)
    hgemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const TcArgs p) {
  using Cfg = TcCfg<BN, STAGES>;
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
      mbar_init(accf_bar(b), 1);                // tcgen05.commit after a tile
      mbar_init(acce_bar(b), Cfg::EPI_WARPS);   // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
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
  // operands and C may come from the previous launch on the stream
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p.num_m, p.num_n, p.group_m, mb, nb);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty)) {
            ok = false;
            break;
          }
          if (!(p.inject == 1 && issued == 0))  // testing aid: withhold one arrival
            mbar_arrive_expect_tx(full_bar(stage), Cfg::STAGE_BYTES);
          tma_load_2d(sA + stage * Cfg::A_BYTES, &tmA, full_bar(stage), kb * Cfg::BK, mb * Cfg::BM);
          tma_load_2d(sB + stage * Cfg::B_BYTES, &tmB, full_bar(stage), kb * Cfg::BK, nb * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last min(issued, STAGES) loads must have landed before the
      // CTA may exit (normally they already have: the MMA warp consumed them).
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
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty)) {
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
          const uint64_t a_desc = sdesc_kmajor_sw128(sA + stage * Cfg::A_BYTES);
          const uint64_t b_desc = sdesc_kmajor_sw128(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k) {
            // +32 bytes per 16-element K step inside the 128-byte swizzle row
            mma_f16_ss(d_tmem, a_desc + 2u * k, b_desc + 2u * k, Cfg::IDESC,
                       (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));  // frees the smem stage once read
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf_bar(acc));  // accumulator complete
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Drain: every MMA issued above completes before TMEM is freed.
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 = tile rows of this warp
    uint8_t* cbuf_base = smem + Cfg::OFF_C + q * Cfg::C_BUFS * Cfg::C_BOX_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cb = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, p.num_m, p.num_n, p.group_m, mb, nb);
      if constexpr (FUSED)
        prefetch_c_row(p.epi, p.C, p.M, p.N, p.ldc, static_cast<int64_t>(mb) * Cfg::BM + q * kEpiRows + lane,
                       static_cast<int64_t>(nb) * BN, BN);
      int ok = 1;
      if (lane == 0) ok = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * Cfg::ACC_COLS);
      const int y0 = mb * Cfg::BM + q * kEpiRows;
#pragma unroll 1
      for (int c = 0; c < BN / kEpiCols; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, v0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        if (c == BN / kEpiCols - 1) {
          // the whole accumulator has been read: hand it back to the MMA warp
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(acc));
        }
        const int x0 = nb * BN + c * kEpiCols;
        if (x0 >= p.N || y0 >= p.M) continue;  // box entirely outside C
        // the store issued from this buffer two boxes ago must have read it
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

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// K = 0: every sum is empty, so C := f(beta·C_old + bias) (alpha·0 = 0), or
// +0 for the plain product.
__global__ void empty_sum_kernel(uint16_t* __restrict__ C, int64_t M, int64_t N, int64_t ldc,
                                 const EpiArgs e) {
  // C and the bias may come from the previous launch on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t count = M * N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const __half* bias = reinterpret_cast<const __half*>(e.bias);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += stride) {
    const int64_t row = i / N, col = i - row * N;
    uint16_t* c = C + row * ldc + col;
    if (e.mode == 0) {
      *c = 0;
      continue;
    }
    const float c_old = e.mode == 2 ? __half2float(__ushort_as_half(*c)) : 0.f;
    const float b = bias ? __half2float(bias[col]) : 0.f;
    *c = __half_as_ushort(__float2half_rn(epi_value(0.f, e, c_old, b)));
  }
}

// Kernels that do nothing, for measuring the fixed cost of a launch: the
// second one with the launch configuration of the pair kernel (clusters of
// two CTAs of 192 threads, its dynamic shared memory).
__global__ void floor_kernel() {}
__global__ void __cluster_dims__(2, 1, 1) floor_pair_kernel() {}

template <typename Kern>
cudaError_t ensure_smem_attr(Kern kern, int bytes, std::atomic<bool>* done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done_per_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done_per_device[dev] = true;
  return e;
}

}  // namespace

cudaError_t launch_tc_128x256(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                              const TcArgs& args, cudaStream_t stream) {
  using Cfg = TcCfg<256, 4>;
  static std::atomic<bool> attr_done[2][64];
  const bool fused = args.epi.mode != 0;
  auto kern = fused ? hgemm_tc_kernel<256, 4, true> : hgemm_tc_kernel<256, 4, false>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::SMEM_BYTES, attr_done[fused ? 1 : 0]);
  if (e != cudaSuccess) return e;
  PdlLaunch l(dim3(static_cast<unsigned>(args.grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, kern, a, b, c, args);
}

cudaError_t launch_tc_128x64(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                             const TcArgs& args, cudaStream_t stream) {
  using Cfg = TcCfg<64, 8>;
  static std::atomic<bool> attr_done[2][64];
  const bool fused = args.epi.mode != 0;
  auto kern = fused ? hgemm_tc_kernel<64, 8, true> : hgemm_tc_kernel<64, 8, false>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::SMEM_BYTES, attr_done[fused ? 1 : 0]);
  if (e != cudaSuccess) return e;
  PdlLaunch l(dim3(static_cast<unsigned>(args.grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, kern, a, b, c, args);
}

cudaError_t launch_floor(int pair_config, int num_sms, int smem_bytes, cudaStream_t stream) {
  if (!pair_config) {
    PdlLaunch l(dim3(1), dim3(32), 0, stream);
    return cudaLaunchKernelEx(&l.cfg, floor_kernel);
  }
  static std::atomic<bool> attr_done[64];
  cudaError_t e = ensure_smem_attr(floor_pair_kernel, smem_bytes, attr_done);
  if (e != cudaSuccess) return e;
  PdlLaunch l(dim3(static_cast<unsigned>(num_sms & ~1)), dim3(192), static_cast<size_t>(smem_bytes), stream);
  return cudaLaunchKernelEx(&l.cfg, floor_pair_kernel);
}

cudaError_t launch_empty_sum(uint16_t* C, int64_t M, int64_t N, int64_t ldc, const EpiArgs& epi,
                             cudaStream_t stream) {
  const int64_t count = M * N;
  int blocks = static_cast<int>((count + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  PdlLaunch l(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream);
  return cudaLaunchKernelEx(&l.cfg, empty_sum_kernel, C, M, N, ldc, epi);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(tc)

}  // namespace hg
