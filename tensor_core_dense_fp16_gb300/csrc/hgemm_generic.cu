// hgemm_generic.cu — C = A·B for operands that TMA cannot describe (a base
// pointer not 16-byte aligned, or K or N not a multiple of 8, so that a row
// pitch is not a multiple of 16 bytes). Any 2-byte-aligned FP16 pointers.
//
// Same arithmetic contract as the other paths: FP16 inputs, FP32
// accumulation on the tensor cores ("GPU架构与CUDA", 混合精度核函数), one
// round-to-nearest-even to FP16. Edge handling follows "GPU架构与CUDA",
// 共享内存与分块: tiles are staged in shared memory with out-of-range elements
// replaced by zero, and only in-range outputs are stored.
//
// Design: one CTA per 128×128 output tile, two CTAs per SM (each one's
// loads, MMAs and epilogue overlap the other's; measured faster than one CTA
// with a deeper ring: the tiles of a triangular product's leaves have few K
// blocks).
//   * warps 0–3 (128 threads) are the loaders: thread t copies row t of the
//     A tile and row t of the B tile for one 64-wide K block with 2-byte loads
//     (bounds-checked, zero outside the matrices) and writes them, 16 bytes
//     at a time, into the same 128-byte-swizzled K-major layout that a TMA
//     copy would produce; a 2-stage ring, one barrier arrival per warp;
//   * warp 8 (one thread) issues tcgen05.mma (M=128, N=128, K=16) into an
//     FP32 accumulator in TMEM;
//   * warps 4–7 read the accumulator with tcgen05.ld, round to FP16 and store
//     each in-range element (C need not be aligned beyond 2 bytes).
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

struct GenCfg {
  static constexpr int BM = 128, BN = 128, BK = 64, STAGES = 2, UMMA_K = 16;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2;  // full, empty, accumulator full, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int LOADER_WARPS = 4;  // warps 0..3; warps 4..7 (epilogue) read TMEM lanes 32·(w%4)
  static constexpr int MMA_WARP = 8;
  static constexpr int THREADS = 9 * 32;
  static constexpr int TMEM_COLS = BN;
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
};

// Row r of a K block (the values of `src` with index in [first, n); zeros
// elsewhere) into the 128-byte-swizzled K-major row r of a shared-memory
// tile. `first` > 0 masks the strictly upper triangle of a triangular operand.
__device__ __forceinline__ void load_row_swizzled(const uint16_t* __restrict__ src, int n, uint8_t* tile,
                                                  int r, int first = 0) {
  uint8_t* row = tile + r * 128;
  if (n == 64 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    // a whole, 16-byte-aligned block: eight vector loads, then the mask
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldg(reinterpret_cast<const uint4*>(src) + j);
    if (first > 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t* w = reinterpret_cast<uint32_t*>(&v[j]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = 8 * j + 2 * u;
          if (k < first) w[u] &= 0xFFFF0000u;
          if (k + 1 < first) w[u] &= 0x0000FFFFu;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) = v[j];
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = 8 * j + 2 * u;
      const uint32_t lo = (k < n && k >= first) ? static_cast<uint32_t>(__ldg(src + k)) : 0u;
      const uint32_t hi = (k + 1 < n && k + 1 >= first) ? static_cast<uint32_t>(__ldg(src + k + 1)) : 0u;
      w[u] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The same row r of a K block for an operand stored with K as its slow
// index: element k at src[k * stride] (k < n; zeros elsewhere). The 2-byte
// loads of a warp's 32 rows are consecutive in memory for each k.
__device__ __forceinline__ void load_row_gather(const uint16_t* __restrict__ src, int64_t stride, int n,
                                                uint8_t* tile, int r) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = 8 * j + 2 * u;
      const uint32_t lo = k < n ? static_cast<uint32_t>(__ldg(src + k * stride)) : 0u;
      const uint32_t hi = k + 1 < n ? static_cast<uint32_t>(__ldg(src + (k + 1) * stride)) : 0u;
      w[u] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One 128×128 tile of C at (m0, n0) over num_kb K blocks. TRI_B: the B
// operand is the lower triangle of a square block (column i of the triangle,
// i.e. operand row gj, holds its values from index gj on), so values at
// k < gj are replaced by zero as they are loaded.
template <bool TRI_B>
__device__ __forceinline__ void generic_tile(const PlainArgs& p, int64_t m0, int64_t n0, int num_kb) {
  using Cfg = GenCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  const uint32_t accf_bar = bar0 + 8u * (2 * Cfg::STAGES);
  const uint32_t drain_bar = accf_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (Cfg::STAGES + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full_bar(s), Cfg::LOADER_WARPS);  // one arrival per loader warp
      mbar_init(empty_bar(s), 1);                 // tcgen05.commit
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == Cfg::MMA_WARP) {
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

  if (warp < Cfg::LOADER_WARPS) {
    // ------------------------------------------------------------ loaders
    const int r = threadIdx.x;  // tile row 0..127
    const int64_t gi = m0 + r, gj = n0 + r;
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = 0; kb < num_kb; ++kb) {
      int ok = 1;
      if (lane == 0) ok = wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int64_t k0 = static_cast<int64_t>(kb) * Cfg::BK;
      const int64_t kn = p.K - k0 < Cfg::BK ? p.K - k0 : Cfg::BK;
      if (p.a_mn)
        load_row_gather(p.A + k0 * p.lda + gi, p.lda, gi < p.M ? static_cast<int>(kn) : 0,
                        smem + Cfg::OFF_A + stage * Cfg::A_BYTES, r);
      else
        load_row_swizzled(p.A + gi * p.lda + k0, gi < p.M ? static_cast<int>(kn) : 0,
                          smem + Cfg::OFF_A + stage * Cfg::A_BYTES, r);
      int first = 0;
      if constexpr (TRI_B) {
        const int64_t f = gj - k0;
        first = f <= 0 ? 0 : (f >= Cfg::BK ? Cfg::BK : static_cast<int>(f));
      }
      if (!TRI_B && p.b_mn)
        load_row_gather(p.B + k0 * p.ldb + gj, p.ldb, gj < p.N ? static_cast<int>(kn) : 0,
                        smem + Cfg::OFF_B + stage * Cfg::B_BYTES, r);
      else
        load_row_swizzled(p.B + gj * p.ldb + k0, gj < p.N ? static_cast<int>(kn) : 0,
                          smem + Cfg::OFF_B + stage * Cfg::B_BYTES, r, first);
      fence_proxy_async_smem();  // generic-proxy writes before tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(stage));
      if (++stage == Cfg::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp == Cfg::MMA_WARP) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!wait_phase(full_bar(stage), phase, wd, kWdMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t a_desc = sdesc_kmajor_sw128(sbase + Cfg::OFF_A + stage * Cfg::A_BYTES);
        const uint64_t b_desc = sdesc_kmajor_sw128(sbase + Cfg::OFF_B + stage * Cfg::B_BYTES);
#pragma unroll
        for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
          mma_f16_ss(tmem_base, a_desc + 2u * k, b_desc + 2u * k, Cfg::IDESC,
                     (kb > 0 || k > 0) ? 1u : 0u);
        mma_commit(empty_bar(stage));
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(accf_bar);
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;
    int ok = 1;
    if (lane == 0) ok = wait_phase(accf_bar, 0, wd, kWdEpiAccFull) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after_sync();
      const int64_t gi = m0 + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < Cfg::BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c * 32, v);
        tmem_ld_wait(v);
        if (gi < p.M) {
          uint16_t* dst = p.C + gi * p.ldc + n0 + c * 32;
          const __half* bias = reinterpret_cast<const __half*>(p.epi.bias);
          if (n0 + c * 32 + 32 <= p.N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 &&
              (p.epi.mode == 0 || (reinterpret_cast<uintptr_t>(bias) & 15u) == 0)) {
            // a whole, aligned 32-column piece of the row: four 16-byte stores
            const int64_t col0 = n0 + c * 32;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 pk;
              if (p.epi.mode == 0) {
                pk.x = pack_half2(v[8 * u], v[8 * u + 1]);
                pk.y = pack_half2(v[8 * u + 2], v[8 * u + 3]);
                pk.z = pack_half2(v[8 * u + 4], v[8 * u + 5]);
                pk.w = pack_half2(v[8 * u + 6], v[8 * u + 7]);
              } else {
                const uint4 c_old = p.epi.mode == 2 ? *reinterpret_cast<const uint4*>(dst + 8 * u)
                                                    : make_uint4(0u, 0u, 0u, 0u);
                pk = epi_pack8(v + 8 * u, p.epi, c_old, load_bias8(p.epi, col0 + 8 * u, p.N));
              }
              *reinterpret_cast<uint4*>(dst + 8 * u) = pk;
            }
            continue;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t col = n0 + c * 32 + j;
            if (col >= p.N) continue;
            float x = __uint_as_float(v[j]);
            if (p.epi.mode != 0)
              x = epi_value(x, p.epi, p.epi.mode == 2 ? __half2float(__ushort_as_half(dst[j])) : 0.f,
                            bias ? __half2float(bias[col]) : 0.f);
            dst[j] = __half_as_ushort(__float2half_rn(x));
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == Cfg::MMA_WARP) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

__global__ void __launch_bounds__(GenCfg::THREADS, 2)
    hgemm_generic_kernel(const PlainArgs p, int tiles_n, int num_kb) {
  generic_tile<false>(p, static_cast<int64_t>(blockIdx.x / tiles_n) * GenCfg::BM,
                      static_cast<int64_t>(blockIdx.x % tiles_n) * GenCfg::BN, num_kb);
}

// The diagonal blocks of a triangular product, one per blockIdx.y: leaf b is
// the product of p's A operand shifted by off columns (M × s) with the lower
// triangle of p's B operand at (off, off) (s × s), into C shifted by off
// columns, where off = leaves.off[b] and s = leaves.size[b].
__global__ void __launch_bounds__(GenCfg::THREADS, 2)
    hgemm_tri_leaves_kernel(const PlainArgs p, const TriLeaves leaves, int tiles_m) {
  const int b = blockIdx.y;
  const int64_t off = leaves.off[b], s = leaves.size[b];
  const int64_t tiles_n = (s + GenCfg::BN - 1) / GenCfg::BN;
  if (static_cast<int64_t>(blockIdx.x) >= tiles_n * tiles_m) return;  // this leaf is narrower
  PlainArgs q = p;
  q.A = p.A + off;
  q.B = p.B + off * p.ldb + off;
  q.C = p.C + off;
  q.N = s;
  q.K = s;
  generic_tile<true>(q, static_cast<int64_t>(blockIdx.x / tiles_n) * GenCfg::BM,
                     static_cast<int64_t>(blockIdx.x % tiles_n) * GenCfg::BN,
                     static_cast<int>((s + GenCfg::BK - 1) / GenCfg::BK));
}

template <typename Kern>
cudaError_t prepare(Kern kern, std::atomic<bool>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GenCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_tri_leaves(const PlainArgs& args, const TriLeaves& leaves, cudaStream_t stream) {
  static std::atomic<bool> attr_done[64];
  cudaError_t e = prepare(hgemm_tri_leaves_kernel, attr_done);
  if (e != cudaSuccess) return e;
  if (leaves.count < 1 || leaves.count > kMaxLeaves) return cudaErrorInvalidValue;
  int64_t widest = 0;
  for (int b = 0; b < leaves.count; ++b) widest = leaves.size[b] > widest ? leaves.size[b] : widest;
  const int64_t tiles_m = (args.M + GenCfg::BM - 1) / GenCfg::BM;
  const int64_t tiles = tiles_m * ((widest + GenCfg::BN - 1) / GenCfg::BN);
  if (tiles > 0x7FFFFFFF || tiles_m > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  PdlLaunch l(dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(leaves.count)), dim3(GenCfg::THREADS),
              GenCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, hgemm_tri_leaves_kernel, args, leaves, static_cast<int>(tiles_m));
}

cudaError_t launch_generic(const PlainArgs& args, int /*num_sms*/, cudaStream_t stream) {
  static std::atomic<bool> attr_done[64];
  cudaError_t e = prepare(hgemm_generic_kernel, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t tiles_n = (args.N + GenCfg::BN - 1) / GenCfg::BN;
  const int64_t tiles = tiles_n * ((args.M + GenCfg::BM - 1) / GenCfg::BM);
  const int64_t num_kb = (args.K + GenCfg::BK - 1) / GenCfg::BK;
  if (tiles > 0x7FFFFFFF || num_kb > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  PdlLaunch l(dim3(static_cast<unsigned>(tiles)), dim3(GenCfg::THREADS), GenCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, hgemm_generic_kernel, args, static_cast<int>(tiles_n),
                            static_cast<int>(num_kb));
}

}  // namespace hg
