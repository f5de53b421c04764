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
// Design: persistent CTAs, two per SM, each walking 128×128 output tiles
// (units) blockIdx.x, blockIdx.x + gridDim.x, ...:
//   * warps 0–3 (128 threads) are the loaders: thread t copies row t of the
//     A tile and row t of the B tile for one 64-wide K block into the same
//     128-byte-swizzled K-major layout that a TMA copy would produce (zero
//     outside the matrices): by asynchronous 16-byte copies (cp.async, two K
//     blocks in flight per thread) when the row starts are 16-byte aligned,
//     else through registers with bounds-checked 2-byte loads (and gathers
//     for M- or N-contiguous operands); a 3-stage ring that runs on across
//     units, one barrier arrival per warp;
//   * warp 8 (one thread) issues tcgen05.mma (M=128, N=128, K=16) into one of
//     two FP32 accumulators in TMEM (2 × 128 columns: two CTAs fill TMEM);
//   * warps 4–7 drain the other accumulator meanwhile with tcgen05.ld, round
//     to FP16 and store each in-range element (C need not be aligned beyond
//     2 bytes).
// The same kernel computes all diagonal blocks of a triangular product in
// one launch (the units of each leaf in turn), masking the upper triangle as
// it loads.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace hg {
namespace {

struct GenCfg {
  static constexpr int BM = 128, BN = 128, BK = 64, STAGES = 3, UMMA_K = 16;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, accumulator full ×2 and empty ×2, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int LOADER_WARPS = 4;  // warps 0..3; warps 4..7 (epilogue) read TMEM lanes 32·(w%4)
  static constexpr int EPI_WARPS = 4;
  static constexpr int MMA_WARP = 8;
  static constexpr int THREADS = 9 * 32;
  static constexpr int TMEM_COLS = 2 * BN;  // two accumulators: two CTAs per SM fill TMEM
  static constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);
  static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM");
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

// Row r of a K block by asynchronous 16-byte copies into the
// 128-byte-swizzled K-major row r of a shared-memory tile: `n` valid values
// from `src` (16-byte aligned), zero-filled past them; chunks of 8 values all
// below `first` (a triangular mask) are zeroed instead of copied. Returns the
// chunk that holds `first` when it is partially masked (its leading
// first - 8·chunk values must be zeroed once the copies have landed), else -1.
__device__ __forceinline__ int issue_row_async(const uint16_t* __restrict__ src, int n, uint8_t* tile, int r,
                                               int first) {
  uint8_t* row = tile + r * 128;
  int fix = -1;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint8_t* dst = row + ((j ^ (r & 7)) << 4);
    int valid = n - 8 * j;
    valid = valid < 0 ? 0 : (valid > 8 ? 8 : valid);
    if (8 * j + 8 <= first) valid = 0;
    if (valid == 0) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    cp_async_16(smem_u32(dst), src + 8 * j, 2 * valid);
    if (8 * j < first) fix = j;
  }
  return fix;
}

// Zeroes the first `count` values of chunk j of swizzled row r.
__device__ __forceinline__ void zero_leading(uint8_t* tile, int r, int j, int count) {
  uint32_t* w = reinterpret_cast<uint32_t*>(tile + r * 128 + ((j ^ (r & 7)) << 4));
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (2 * u + 1 < count)
      w[u] = 0u;
    else if (2 * u < count)
      w[u] &= 0xFFFF0000u;
  }
}

// A K block whose copies are in flight: its ring stage and the chunk of its
// B row a triangular mask must still fix (-1: none).
struct PendingBlock {
  int stage;
  int fix_j;
  int fix_cnt;
};

// Work unit t of a launch: the 128×128 tile of C at (m0, n0) over num_kb K
// blocks, with the operands it reads. Units are numbered tile by tile, N
// tiles fastest (neighbouring units share their rows of A); for the leaves of
// a triangular product, leaf b owns units [b·tiles_m·tiles_n, (b+1)·…) with
// its operands shifted to the leaf, and a narrower leaf's missing N tiles are
// empty units that every role skips alike.
struct GenUnit {
  PlainArgs q;
  int64_t m0, n0;
  int num_kb;
  bool valid;
};

template <bool TRI_B>
__device__ __forceinline__ GenUnit gen_unit(const PlainArgs& p, const TriLeaves& leaves, int64_t t,
                                            int64_t tiles_m, int64_t tiles_n) {
  using Cfg = GenCfg;
  GenUnit u;
  const int64_t per = tiles_m * tiles_n;
  const int64_t b = t / per, r = t - b * per;
  const int64_t mt = r / tiles_n, nt = r - mt * tiles_n;
  u.q = p;
  if constexpr (TRI_B) {
    const int64_t off = leaves.off[b], s = leaves.size[b];
    u.q.A = p.A + off;
    u.q.B = p.B + off * p.ldb + off;
    u.q.C = p.C + off;
    u.q.N = s;
    u.q.K = s;
  }
  u.m0 = mt * Cfg::BM;
  u.n0 = nt * Cfg::BN;
  u.valid = u.n0 < u.q.N && u.m0 < u.q.M;
  u.num_kb = static_cast<int>((u.q.K + Cfg::BK - 1) / Cfg::BK);
  return u;
}

// A persistent CTA: units blockIdx.x, blockIdx.x + gridDim.x, ... The loader
// warps keep the operand ring going across units, the MMA warp fills one of
// two TMEM accumulators while the epilogue drains the other. TRI_B: the B
// operand of each unit is the lower triangle of a square block (column i of
// the triangle, i.e. operand row gj, holds its values from index gj on), so
// values at k < gj are replaced by zero as they are loaded.
template <bool TRI_B>
__device__ __forceinline__ void generic_units(const PlainArgs& p, const TriLeaves& leaves, int64_t units,
                                              int64_t tiles_m, int64_t tiles_n) {
  using Cfg = GenCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Cfg::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (Cfg::STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * Cfg::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * Cfg::STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full_bar(s), Cfg::LOADER_WARPS);  // one arrival per loader warp
      mbar_init(empty_bar(s), 1);                 // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);               // tcgen05.commit
      mbar_init(acce_bar(b), Cfg::EPI_WARPS);  // one arrival per epilogue warp
    }
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
    // Rows with 16-byte aligned starts (K-contiguous operand, aligned base
    // and pitch) go by asynchronous copies, kInFlight K blocks in flight per
    // thread: a block is published (fence to the async proxy, one arrival
    // per warp) once its copies have landed and a triangular mask has
    // zeroed its leading values. Other rows go through registers.
    constexpr int kInFlight = Cfg::STAGES - 1;
    const int r = threadIdx.x;  // tile row 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    static_assert(kInFlight == 2, "two pending blocks: older and newer");
    PendingBlock older{0, -1, 0}, newer{0, -1, 0};
    int npend = 0;
    // the older pending block: its copies are complete (the caller waited)
    auto publish_oldest = [&]() {
      if (older.fix_j >= 0)
        zero_leading(smem + Cfg::OFF_B + older.stage * Cfg::B_BYTES, r, older.fix_j, older.fix_cnt);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(older.stage));
      older = newer;
      --npend;
    };
    for (int64_t t = blockIdx.x; ok && t < units; t += gridDim.x) {
      const GenUnit u = gen_unit<TRI_B>(p, leaves, t, tiles_m, tiles_n);
      if (!u.valid) continue;
      const int64_t gi = u.m0 + r, gj = u.n0 + r;
      const bool a_async = !u.q.a_mn && ((reinterpret_cast<uintptr_t>(u.q.A) & 15u) == 0) && u.q.lda % 8 == 0;
      const bool b_async = (TRI_B || !u.q.b_mn) && ((reinterpret_cast<uintptr_t>(u.q.B) & 15u) == 0) &&
                           u.q.ldb % 8 == 0;
      for (int kb = 0; kb < u.num_kb; ++kb) {
        int good = 1;
        if (lane == 0) good = wait_phase(empty_bar(stage), phase ^ 1u, wd, kWdProducerEmpty) ? 1 : 0;
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        const int64_t k0 = static_cast<int64_t>(kb) * Cfg::BK;
        const int64_t kn = u.q.K - k0 < Cfg::BK ? u.q.K - k0 : Cfg::BK;
        uint8_t* sa = smem + Cfg::OFF_A + stage * Cfg::A_BYTES;
        uint8_t* sb = smem + Cfg::OFF_B + stage * Cfg::B_BYTES;
        const int na = gi < u.q.M ? static_cast<int>(kn) : 0;
        const int nb = gj < u.q.N ? static_cast<int>(kn) : 0;
        (void)HG_DBG_INDEX(k0 + kn - 1, u.q.K);
        if (u.q.a_mn)
          load_row_gather(u.q.A + k0 * u.q.lda + gi, u.q.lda, na, sa, r);
        else if (a_async)
          issue_row_async(u.q.A + gi * u.q.lda + k0, na, sa, r, 0);
        else
          load_row_swizzled(u.q.A + gi * u.q.lda + k0, na, sa, r);
        int first = 0;
        if constexpr (TRI_B) {
          const int64_t f = gj - k0;
          first = f <= 0 ? 0 : (f >= Cfg::BK ? Cfg::BK : static_cast<int>(f));
        }
        PendingBlock b{stage, -1, 0};
        if (!TRI_B && u.q.b_mn) {
          load_row_gather(u.q.B + k0 * u.q.ldb + gj, u.q.ldb, nb, sb, r);
        } else if (b_async) {
          const int fj = issue_row_async(u.q.B + gj * u.q.ldb + k0, nb, sb, r, first);
          if (fj >= 0) {
            b.fix_j = fj;
            b.fix_cnt = first - 8 * fj;
          }
        } else {
          load_row_swizzled(u.q.B + gj * u.q.ldb + k0, nb, sb, r, first);
        }
        cp_async_commit();
        if (npend == 0)
          older = b;
        else
          newer = b;
        ++npend;
        if (npend == kInFlight) {
          cp_async_wait<kInFlight - 1>();
          publish_oldest();
        }
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // the blocks still in flight (after a failed wait too: their copies must
    // land before the CTA's shared memory goes away)
    cp_async_wait<0>();
    while (npend > 0) publish_oldest();
  } else if (warp == Cfg::MMA_WARP) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < units; t += gridDim.x) {
        const GenUnit u = gen_unit<TRI_B>(p, leaves, t, tiles_m, tiles_n);
        if (!u.valid) continue;
        // the epilogue must have drained this accumulator's previous tile
        if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, wd, kWdMmaAccEmpty)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::BN);
        for (int kb = 0; kb < u.num_kb; ++kb) {
          if (!wait_phase(full_bar(stage), phase, wd, kWdMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = sdesc_kmajor_sw128(sbase + Cfg::OFF_A + stage * Cfg::A_BYTES);
          const uint64_t b_desc = sdesc_kmajor_sw128(sbase + Cfg::OFF_B + stage * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k)
            mma_f16_ss(d_tmem, a_desc + 2u * k, b_desc + 2u * k, Cfg::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty_bar(stage));
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0, wd);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < units; t += gridDim.x) {
      const GenUnit u = gen_unit<TRI_B>(p, leaves, t, tiles_m, tiles_n);
      if (!u.valid) continue;
      int ok = 1;
      if (lane == 0) ok = wait_phase(accf_bar(acc), acc_phase, wd, kWdEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const int64_t gi = u.m0 + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * Cfg::BN);
      const PlainArgs& c = u.q;
#pragma unroll 1
      for (int ch = 0; ch < Cfg::BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + ch * 32, v);
        tmem_ld_wait(v);
        if (gi >= c.M) continue;
        uint16_t* dst = c.C + gi * c.ldc + u.n0 + ch * 32;
        const __half* bias = reinterpret_cast<const __half*>(c.epi.bias);
        if (u.n0 + ch * 32 + 32 <= c.N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 &&
            (c.epi.mode == 0 || (reinterpret_cast<uintptr_t>(bias) & 15u) == 0)) {
          // a whole, aligned 32-column piece of the row: four 16-byte stores
          const int64_t col0 = u.n0 + ch * 32;
          if (!HG_DBG_INDEX(gi, c.M) || !HG_DBG_INDEX(col0 + 31, c.N) || !HG_DBG_ALIGN(dst, 16)) continue;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 pk;
            if (c.epi.mode == 0) {
              pk.x = pack_half2(v[8 * w], v[8 * w + 1]);
              pk.y = pack_half2(v[8 * w + 2], v[8 * w + 3]);
              pk.z = pack_half2(v[8 * w + 4], v[8 * w + 5]);
              pk.w = pack_half2(v[8 * w + 6], v[8 * w + 7]);
            } else {
              const uint4 c_old = c.epi.mode == 2 ? *reinterpret_cast<const uint4*>(dst + 8 * w)
                                                  : make_uint4(0u, 0u, 0u, 0u);
              pk = epi_pack8(v + 8 * w, c.epi, c_old, load_bias8(c.epi, col0 + 8 * w, c.N));
            }
            *reinterpret_cast<uint4*>(dst + 8 * w) = pk;
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t col = u.n0 + ch * 32 + j;
          if (col >= c.N) continue;
          float x = __uint_as_float(v[j]);
          if (c.epi.mode != 0)
            x = epi_value(x, c.epi, c.epi.mode == 2 ? __half2float(__ushort_as_half(dst[j])) : 0.f,
                          bias ? __half2float(bias[col]) : 0.f);
          dst[j] = __half_as_ushort(__float2half_rn(x));
        }
      }
      // this accumulator may be overwritten by the unit after next
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == Cfg::MMA_WARP) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

__global__ void __launch_bounds__(GenCfg::THREADS, 2)
    hgemm_generic_kernel(const PlainArgs p, int64_t tiles_m, int64_t tiles_n) {
  const TriLeaves none{};
  generic_units<false>(p, none, tiles_m * tiles_n, tiles_m, tiles_n);
}

// The diagonal blocks of a triangular product: leaf b is the product of p's
// A operand shifted by off columns (M × s) with the lower triangle of p's B
// operand at (off, off) (s × s), into C shifted by off columns, where
// off = leaves.off[b] and s = leaves.size[b]; tiles_n covers the widest leaf.
__global__ void __launch_bounds__(GenCfg::THREADS, 2)
    hgemm_tri_leaves_kernel(const PlainArgs p, const TriLeaves leaves, int64_t tiles_m, int64_t tiles_n) {
  generic_units<true>(p, leaves, leaves.count * tiles_m * tiles_n, tiles_m, tiles_n);
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

// Persistent grid: two CTAs per SM, or one per unit when there are fewer.
unsigned persistent_grid(int64_t units, int num_sms) {
  const int64_t slots = 2 * static_cast<int64_t>(num_sms > 0 ? num_sms : 1);
  return static_cast<unsigned>(units < slots ? (units > 0 ? units : 1) : slots);
}

}  // namespace

cudaError_t launch_tri_leaves(const PlainArgs& args, const TriLeaves& leaves, int num_sms, cudaStream_t stream) {
  static std::atomic<bool> attr_done[64];
  cudaError_t e = prepare(hgemm_tri_leaves_kernel, attr_done);
  if (e != cudaSuccess) return e;
  if (leaves.count < 1 || leaves.count > kMaxLeaves) return cudaErrorInvalidValue;
  int64_t widest = 0;
  for (int b = 0; b < leaves.count; ++b) widest = leaves.size[b] > widest ? leaves.size[b] : widest;
  const int64_t tiles_m = (args.M + GenCfg::BM - 1) / GenCfg::BM;
  const int64_t tiles_n = (widest + GenCfg::BN - 1) / GenCfg::BN;
  PdlLaunch l(dim3(persistent_grid(leaves.count * tiles_m * tiles_n, num_sms)), dim3(GenCfg::THREADS),
              GenCfg::SMEM_BYTES, stream);
  return cudaLaunchKernelEx(&l.cfg, hgemm_tri_leaves_kernel, args, leaves, tiles_m, tiles_n);
}

cudaError_t launch_generic(const PlainArgs& args, int num_sms, cudaStream_t stream) {
  static std::atomic<bool> attr_done[64];
  cudaError_t e = prepare(hgemm_generic_kernel, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t tiles_n = (args.N + GenCfg::BN - 1) / GenCfg::BN;
  const int64_t tiles_m = (args.M + GenCfg::BM - 1) / GenCfg::BM;
  PdlLaunch l(dim3(persistent_grid(tiles_m * tiles_n, num_sms)), dim3(GenCfg::THREADS), GenCfg::SMEM_BYTES,
              stream);
  return cudaLaunchKernelEx(&l.cfg, hgemm_generic_kernel, args, tiles_m, tiles_n);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(generic)

}  // namespace hg
