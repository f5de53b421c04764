// hgemm_trsm.cu — the pieces of the triangular solve of
// "异构计算中高性能TRMM与TRSM的递归算法实现" (§2.3) that are not products: the
// scaled copy of the right-hand side, the solve of one diagonal block (order
// ≤ 256) for all right-hand sides, and, for the entry points with a
// workspace, the inverses of all diagonal blocks of order ≤ 512 (the same
// solve against the columns of the identity, one warp per 32 rows). The
// recursion, its GEMM updates and the products by the inverses are in
// hgemm_api.cu.
//
// The system solved, in the variant of the page's §2.2 product (left side,
// lower triangle, transposed): Aᵀ·X = alpha·B, every matrix column-major
// (A(r,c) at A[c·lda + r], X(r,j) at X[j·ldx + r]). Row i of the system is
//   Σ_{k ≥ i} A(k,i)·x_k = b_i,
// so the block is solved by back substitution, last row first.
//
// Leaf solve (§2.3: the right-hand sides spread over thread blocks, a light
// barrier between steps): warp w of a block owns rows 32w .. 32w+31 of the
// diagonal block for COLS right-hand sides, in registers (the accumulator
// fragments of the tensor-core update below). The rows are taken in groups
// of 32 (one warp's rows), last group first. A group's own 32×32 triangle
// L_g is applied through its inverse, which warp g computes in FP32 at the
// start (forward substitution on the columns of the identity), so that the
// group's solution x_g = (L_g⁻¹)ᵀ·b_g is a small product spread over all
// threads, not a chain of 32 dependent steps in one warp. Per group: the
// owning warp publishes its b, barrier, all threads form x_g (FP32),
// barrier, and every warp above the group subtracts Σ_c A(c,r)·x_c over the
// group's rows on the tensor cores (mma.sync m16n8k16: A(c0 .. c0+31, r),
// contiguous in the column-major A, copied a group ahead into shared memory
// and read back with ldmatrix; x_g rounded to FP16, as the recursion's GEMM updates see
// X; FP32 accumulators holding the right-hand sides). The solution is
// rounded once to FP16.
//
// The page's literal orientation (FWD, §2.3: X = A\B): A·X = alpha·B with
// the same lower A, untransposed. Row i is Σ_{k ≤ i} A(i,k)·x_k = b_i, so
// the block is solved by forward substitution: the groups go first to last,
// each applied through the inverse of its diagonal triangle (warp g computes
// the rows of L_g⁻¹ by back substitution on the columns of L_g, so that
// x_g = L_g⁻¹·b_g is the same small product), and the warps below the group
// subtract Σ_c A(r,c)·x_c: A(r0 .. r0+31, c) is contiguous for each of the
// group's columns c, so each warp stages its own rows of the group's 32
// columns (k-major, a group ahead) and reads them back transposed with
// ldmatrix.trans as the same m16k16 fragments.
//
// Launch overlap: the inverses only read A, which no launch of the solve
// writes, so they are computed before the kernel waits for the previous
// launch on the stream (griddepcontrol.wait) and read X.
#include <atomic>

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace hg {
namespace {

constexpr int kLeafMax = kTrsmLeaf;                     // largest diagonal block solved per right-hand side
constexpr int kMaxDevices = 64;
constexpr int kGroup = 32;                  // rows per barrier step: one warp's rows

// Row pitch (floats) of the published b and x rows: the padding puts
// consecutive lanes' 16-byte accesses in different banks.
template <int COLS>
__host__ __device__ constexpr int pub_pitch() {
  return COLS + 4;
}

// Halves per column of the FP16 copy of -x_g (the mma B operand): the
// padding spreads a warp's 32-bit fragment loads over all banks.
constexpr int KP = kGroup + 8;

// Halves per row of the staged A segments (32 values + 8 of padding: the
// 80-byte pitch puts the 8 rows of an ldmatrix load in different banks).
constexpr int AP = kGroup + 8;

// LEAF: the largest block order the kernel takes (one warp per 32 rows).
template <int COLS, int LEAF = kLeafMax>
constexpr int leaf_smem() {
  return (LEAF / kGroup) * kGroup * kGroup * 4 + 2 * kGroup * pub_pitch<COLS>() * 4 + COLS * KP * 2 +
         2 * LEAF * AP * 2;
}
// Halves per k-row of the forward solve's staged columns: the block's rows
// plus 8 of padding (the 8 k-rows of an ldmatrix load land in different banks).
template <int LEAF>
constexpr int fwd_pitch() {
  return LEAF + 8;
}
static_assert(2 * kGroup * fwd_pitch<kLeafMax>() <= 2 * kLeafMax * AP, "the forward stage fits in the same space");

// The m16k16 A fragment of mma.sync from a row-major 16×16 FP16 tile in
// shared memory: lane l gives the address of row (l % 8) + 8·((l / 8) % 2),
// columns 8·(l / 16) .. +7.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  if (!HG_DBG_SMEM(addr, 16)) return;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// The same fragment from a 16×16 tile stored transposed (k-major: 16 rows of
// k, each 16 contiguous row values): lane l gives the address of k-row
// (l % 8) + 8·(l / 16), row values 8·((l / 8) % 2) .. +7.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  if (!HG_DBG_SMEM(addr, 16)) return;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// mma.sync m16n8k16, FP16 operands, FP32 accumulator in place: d += a·b.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A(row0 + q, col) for q < 32 (q < valid; 0 past it), packed as 32 halves.
__device__ __forceinline__ void load_col32(const uint16_t* __restrict__ A, int64_t lda, int64_t col,
                                           int64_t row0, int valid, bool vec, uint4 (&out)[4]) {
  const uint16_t* src = A + col * lda + row0;
  if (vec && valid == kGroup) {
#pragma unroll
    for (int p = 0; p < 4; ++p) out[p] = __ldg(reinterpret_cast<const uint4*>(src) + p);
  } else {
    uint32_t w[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const uint32_t lo = 2 * p < valid ? src[2 * p] : 0u;
      const uint32_t hi = 2 * p + 1 < valid ? src[2 * p + 1] : 0u;
      w[p] = lo | (hi << 16);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) out[p] = make_uint4(w[4 * p], w[4 * p + 1], w[4 * p + 2], w[4 * p + 3]);
  }
}

// Half q of a packed column segment, as FP32.
__device__ __forceinline__ float col32_at(const uint4 (&v)[4], int q) {
  const uint4 c = v[q / 8];
  const uint32_t w = (q % 8) < 2 ? c.x : (q % 8) < 4 ? c.y : (q % 8) < 6 ? c.z : c.w;
  return __half2float(__ushort_as_half(static_cast<uint16_t>(w >> (16 * (q & 1)))));
}

// The solve of the diagonal block A(off .. off+s-1, off .. off+s-1) for the
// right-hand sides j0 .. j0+COLS-1, rows xoff .. xoff+s-1 of X, in place.
// identity: the right-hand sides are the columns of the identity (X is not
// read), so the block computes columns j0.. of the inverse of the block's
// transpose.
// FWD: the literal orientation A·X = B (forward substitution); otherwise
// Aᵀ·X = B (back substitution).
template <int COLS, int LEAF, bool FWD = false>
__device__ __forceinline__ void trsm_leaf_body(const uint16_t* __restrict__ A, int64_t lda,
                                               uint16_t* __restrict__ X, int64_t ldx, int64_t off,
                                               int64_t xoff, int s, int64_t m, int chained, bool identity,
                                               int64_t j0) {
  extern __shared__ __align__(16) uint8_t smem[];
  if (!chained) grid_dependency_wait();
  // diag[g][k][j]: first L_g(k, j) in FP32 (L_g the diagonal triangle of
  // rows 32g .. 32g+31), then, in place, (L_g⁻¹)(k, j)
  float* diag = reinterpret_cast<float*>(smem);
  constexpr int P = pub_pitch<COLS>();
  float* pub_b = diag + (LEAF / kGroup) * kGroup * kGroup;  // [kGroup][P]: b of the group's rows
  float* pub_x = pub_b + kGroup * P;                // [kGroup][P]: x of the group's rows
  __half* pub_xh = reinterpret_cast<__half*>(pub_x + kGroup * P);  // [COLS][KP]: -x_g in FP16
  // [2][LEAF][AP]: A(c0 .. c0+31, r) of a group, row r of the block,
  // double-buffered (the next group's segments arrive during this group)
  uint16_t* a_stage = reinterpret_cast<uint16_t*>(pub_xh + COLS * KP);
  const int r = threadIdx.x;
  const int lane = r & 31, warp = r >> 5;
  const int groups = (s + kGroup - 1) / kGroup;  // the block's warps (warps past them only synchronise)
  // 16-byte loads of A's column segments: column starts 16-byte aligned
  const bool vec = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && (lda % 8) == 0 && (off % 8) == 0;

  // Warp g: the inverse of its diagonal triangle L_g. Lane i loads column i
  // of L_g, stores it transposed (rows of L_g contiguous, FP32), then
  // computes column i of L_g⁻¹ by forward substitution on e_i, reading rows
  // of L_g 16 bytes at a time (lane k supplies 1/L_g(k,k) by shuffle, off the
  // dependent chain), and overwrites L_g with it. Entries above the diagonal
  // are loaded but never read; rows and columns past the block's order are 0.
  {
    const int g = warp, c0 = g * kGroup, sg = min(kGroup, s - c0);
    float* blk = diag + g * kGroup * kGroup;
    if (lane < sg) {
      uint4 col[4];
      load_col32(A, lda, off + c0 + lane, off + c0, sg, vec, col);
#pragma unroll
      for (int k = 0; k < kGroup; ++k) blk[k * kGroup + lane] = col32_at(col, k);
    }
    __syncwarp();
    const float rd_own = lane < sg ? 1.0f / blk[lane * kGroup + lane] : 0.f;
    float mcol[kGroup];
    if constexpr (!FWD) {
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const float4* rowv = reinterpret_cast<const float4*>(blk + k * kGroup);
        const float rd = __shfl_sync(0xffffffffu, rd_own, k);
        float acc = (k == lane) ? 1.0f : 0.0f;
#pragma unroll
        for (int j4 = 0; j4 < (k + 3) / 4; ++j4) {
          const float4 l = rowv[j4];
          if (4 * j4 + 0 < k) acc = fmaf(-l.x, mcol[4 * j4 + 0], acc);
          if (4 * j4 + 1 < k) acc = fmaf(-l.y, mcol[4 * j4 + 1], acc);
          if (4 * j4 + 2 < k) acc = fmaf(-l.z, mcol[4 * j4 + 2], acc);
          if (4 * j4 + 3 < k) acc = fmaf(-l.w, mcol[4 * j4 + 3], acc);
        }
        mcol[k] = (k < sg && k >= lane) ? acc * rd : 0.f;
      }
    } else {
      // row `lane` of L_g⁻¹: y with L_gᵀ·y = e_lane, by back substitution on
      // the columns of L_g (every lane reads the same entry: a broadcast);
      // its entries past the lane's own index are zero
#pragma unroll
      for (int k = kGroup - 1; k >= 0; --k) {
        const float rd = __shfl_sync(0xffffffffu, rd_own, k);
        float acc = (k == lane) ? 1.0f : 0.0f;
#pragma unroll
        for (int j = k + 1; j < kGroup; ++j) acc = fmaf(-blk[j * kGroup + k], mcol[j], acc);
        mcol[k] = (k < sg && k <= lane) ? acc * rd : 0.f;
      }
    }
    __syncwarp();
    // L_g⁻¹ in place: (transposed) blk[k][i] = L_g⁻¹(k, i), column `lane`;
    // (forward) blk[k][i] = L_g⁻¹(i, k), row `lane`. Either way step (2)
    // below reads blk[k][lane].
#pragma unroll
    for (int k = 0; k < kGroup; ++k) blk[k * kGroup + lane] = lane < sg ? mcol[k] : 0.f;
  }

  // The rows above a group take its update on the tensor cores: b (rows ×
  // right-hand sides) -= A_g (rows × the group's 32 rows) · x_g, as
  // mma.sync m16n8k16 products (FP16 operands, FP32 accumulation) whose
  // accumulators are the b values themselves. Warp w holds its 32 rows as
  // c[mt][nt][e]: row 16·mt + gid (+8 for e ≥ 2) of the warp's rows, column
  // 8·nt + 2·tig (+1 for odd e), gid = lane / 4, tig = lane % 4 (the
  // accumulator layout of that instruction).
  constexpr int NT = COLS / 8;
  const int gid = lane >> 2, tig = lane & 3;
  float c[2][NT][4];
  // X comes from the previous launch on the stream: everything above only
  // read A, which no launch of the solve writes (a chained launch starts only
  // after its predecessor passed its own wait, so work enqueued before the
  // solve is complete). The first launch of a solve waits before reading A.
  grid_dependency_wait();
  grid_launch_dependents();
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = warp * kGroup + 16 * mt + gid + (e >= 2 ? 8 : 0);
        const int64_t j = j0 + 8 * nt + 2 * tig + (e & 1);
        c[mt][nt][e] = (row < s && j < m)
                           ? (identity ? (row == j ? 1.f : 0.f) : __half2float(__ushort_as_half(X[j * ldx + xoff + row])))
                           : 0.f;
      }
  // 32-bit loads of A's K pairs: A 4-byte aligned and lda even (off is a
  // multiple of 64)
  const bool pairs = ((reinterpret_cast<uintptr_t>(A) & 3u) == 0) && (lda % 2) == 0;
  // A's column segments staged by asynchronous 16-byte copies, a group ahead:
  // A 16-byte aligned and lda a multiple of 8
  const bool staged = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && (lda % 8) == 0;
  // warps that take group g's update: above it (transposed), or below it
  // among the block's warps (forward)
  auto updates = [&](int w, int g) { return FWD ? (w > g && w < groups) : (w < g); };
  constexpr int FPITCH = fwd_pitch<LEAF>();
  // forward: warp w's rows of group g's columns, A(off+32w .. +31, off+32g+k)
  // for k < 32 (each contiguous), k-major into buffer g % 2, zero past the
  // block's order (rows and columns)
  auto stage_fwd = [&](int g) {
    if (!updates(warp, g)) return;
    const int c0 = g * kGroup, sg = min(kGroup, s - c0);
    uint16_t* buf = a_stage + (g & 1) * kGroup * FPITCH;
#pragma unroll
    for (int i = lane; i < kGroup * 4; i += 32) {
      const int k = i >> 2, row = warp * kGroup + 8 * (i & 3);
      int valid = s - row;
      valid = valid < 0 ? 0 : (valid > 8 ? 8 : valid);
      uint16_t* dst = buf + k * FPITCH + row;
      // the group's columns and the warp's rows stay inside the block
      if (valid > 0 && k < sg && (!HG_DBG_INDEX(c0 + k, s) || !HG_DBG_INDEX(row + valid - 1, s))) continue;
      if (k < sg && valid > 0)
        cp_async_16(smem_u32(dst), A + (off + c0 + k) * lda + off + row, 2 * valid);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // the warp's rows' segments of group g: A(off+32g .. +31, off+rr) for its
  // rows rr, zero past the block's order, into buffer g % 2 (warps above
  // group g only). Each segment is 64 contiguous bytes of A, copied by four
  // consecutive lanes, so that one copy instruction of the warp touches 8
  // segments rather than 32 (the copies' cost is in the lines they touch).
  auto stage_group = [&](int g) {
    if constexpr (FWD) {
      stage_fwd(g);
      return;
    }
    if (warp >= g) return;
    const int c0 = g * kGroup, sg = min(kGroup, s - c0);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int i = it * 32 + lane;
      const int rr = warp * kGroup + (i >> 2), q = i & 3;
      int valid = sg - 8 * q;
      valid = valid < 0 ? 0 : (valid > 8 ? 8 : valid);
      uint16_t* dst = a_stage + ((g & 1) * LEAF + rr) * AP + 8 * q;
      if (valid > 0)
        cp_async_16(smem_u32(dst), A + (off + rr) * lda + off + c0 + 8 * q, 2 * valid);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // Against the identity, the right-hand sides j0 .. j0+COLS-1 have zero
  // solutions past the last of them (transposed: the inverse of Lᵀ is upper
  // triangular) or before the first (forward: L⁻¹ is lower triangular); the
  // groups holding only such rows have b = 0, so x_g = 0 and their updates
  // change nothing: they are skipped (their rows keep the identity's 0).
  int g_begin = FWD ? 0 : groups - 1, steps = groups;
  if (identity) {
    if constexpr (FWD) {
      g_begin = static_cast<int>(j0 / kGroup);
      steps = groups - g_begin;
    } else {
      const int64_t last = (j0 + COLS - 1) / kGroup;
      g_begin = last < groups - 1 ? static_cast<int>(last) : groups - 1;
      steps = g_begin + 1;
    }
  }
  if (staged && steps > 0) stage_group(g_begin);
  cp_async_commit();

  for (int gi = 0; gi < steps; ++gi) {
    const int g = FWD ? g_begin + gi : g_begin - gi;  // forward: first group first; else last first
    const int c0 = g * kGroup, sg = min(kGroup, s - c0);
    // A's values for this warp's update, loaded now to land while the group
    // is solved: af[mt][ks] is the m16k16 fragment of rows 16·mt.. of the
    // warp and the group's rows 16·ks.., i.e. A(c0 + k, r) (contiguous in k)
    uint32_t af[2][2][4] = {};
    // one copy group per step: the next group's segments
    const int gn = FWD ? g + 1 : g - 1;
    if (staged && gn >= 0 && gn < groups) {
      __syncwarp();  // this warp's reads of the buffer (two groups ago) are done
      stage_group(gn);
    }
    cp_async_commit();
    if (!staged && updates(warp, g)) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = warp * kGroup + 16 * mt + gid + ((e & 1) ? 8 : 0);  // row in the block
            const int k = 16 * ks + 2 * tig + ((e & 2) ? 8 : 0);
            if constexpr (FWD) {
              // A(off + rr, off + c0 + k) and the next column: lda apart
              const uint16_t* src = A + (off + c0 + k) * lda + off + rr;
              const uint32_t lo = (k < sg && rr < s) ? src[0] : 0u;
              const uint32_t hi = (k + 1 < sg && rr < s) ? src[lda] : 0u;
              af[mt][ks][e] = lo | (hi << 16);
            } else {
              const uint16_t* src = A + (off + rr) * lda + off + c0 + k;
              if (pairs && k + 1 < sg) {
                af[mt][ks][e] = __ldg(reinterpret_cast<const unsigned int*>(src));
              } else {
                const uint32_t lo = k < sg ? src[0] : 0u;
                const uint32_t hi = k + 1 < sg ? src[1] : 0u;
                af[mt][ks][e] = lo | (hi << 16);
              }
            }
          }
    }
    // (1) the owning warp's rows, complete with every later group's update
    if (warp == g) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float* d = pub_b + (16 * mt + gid) * P + 8 * nt + 2 * tig;
          *reinterpret_cast<float2*>(d) = make_float2(c[mt][nt][0], c[mt][nt][1]);
          *reinterpret_cast<float2*>(d + 8 * P) = make_float2(c[mt][nt][2], c[mt][nt][3]);
        }
    }
    // This barrier also orders the group's writes of the published rows after
    // every read of them for the previous group, and (first time round) the
    // inverses before their use by other warps.
    __syncthreads();
    // (2) x_g(i, jj) = Σ_k L_g⁻¹(k, i)·b_g(k, jj): lane i, four right-hand
    // sides per thread (jj = 4q .. 4q+3 for q = warp, warp + groups, ...);
    // also -x_g in FP16, column by column, as the mma B operand
    {
      const float* mi = diag + g * kGroup * kGroup + lane;
      for (int q = warp; warp < groups && q < COLS / 4; q += groups) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          const float mk = mi[k * kGroup];
          const float4 bk = *reinterpret_cast<const float4*>(pub_b + k * P + 4 * q);
          acc.x = fmaf(mk, bk.x, acc.x);
          acc.y = fmaf(mk, bk.y, acc.y);
          acc.z = fmaf(mk, bk.z, acc.z);
          acc.w = fmaf(mk, bk.w, acc.w);
        }
        *reinterpret_cast<float4*>(pub_x + lane * P + 4 * q) = acc;
        pub_xh[(4 * q + 0) * KP + lane] = __float2half_rn(-acc.x);
        pub_xh[(4 * q + 1) * KP + lane] = __float2half_rn(-acc.y);
        pub_xh[(4 * q + 2) * KP + lane] = __float2half_rn(-acc.z);
        pub_xh[(4 * q + 3) * KP + lane] = __float2half_rn(-acc.w);
      }
    }
    __syncthreads();
    if (warp == g) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float* x = pub_x + (16 * mt + gid) * P + 8 * nt + 2 * tig;
          const float2 lo = *reinterpret_cast<const float2*>(x);
          const float2 hi = *reinterpret_cast<const float2*>(x + 8 * P);
          c[mt][nt][0] = lo.x;
          c[mt][nt][1] = lo.y;
          c[mt][nt][2] = hi.x;
          c[mt][nt][3] = hi.y;
        }
    } else if (updates(warp, g)) {
      // (3) rows above (below, forward) the group: b += A_g · (-x_g) (A = 0
      // past the block's order)
      if (staged) {
        cp_async_wait<1>();  // this group's segments (the next group's may be in flight)
        __syncwarp();
        if constexpr (FWD) {
          const uint16_t* base = a_stage + (g & 1) * kGroup * FPITCH + warp * kGroup;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const int k = 16 * ks + (lane & 7) + ((lane >> 4) << 3);
              const int row = 16 * mt + ((lane >> 3) & 1) * 8;
              ldmatrix_x4_trans(af[mt][ks], smem_u32(base + k * FPITCH + row));
            }
        } else {
          const uint16_t* base = a_stage + ((g & 1) * LEAF + warp * kGroup) * AP;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const int row = 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
              ldmatrix_x4(af[mt][ks], smem_u32(base + row * AP + 16 * ks + (lane >> 4) * 8));
            }
        }
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const __half* xb = pub_xh + (8 * nt + gid) * KP + 16 * ks + 2 * tig;
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xb);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xb + 8);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) mma_16816(c[mt][nt], af[mt][ks], b0, b1);
        }
    }
  }

#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = warp * kGroup + 16 * mt + gid + (e >= 2 ? 8 : 0);
        const int64_t j = j0 + 8 * nt + 2 * tig + (e & 1);
        if (row < s && j < m) X[j * ldx + xoff + row] = __half_as_ushort(__float2half_rn(c[mt][nt][e]));
      }
}

template <int COLS, bool FWD>
__global__ void __launch_bounds__(kLeafMax, 2)
    trsm_leaf_kernel(const uint16_t* __restrict__ A, int64_t lda, uint16_t* __restrict__ X,
                     int64_t ldx, int64_t off, int s, int64_t m, int chained) {
  trsm_leaf_body<COLS, kLeafMax, FWD>(A, lda, X, ldx, off, off, s, m, chained, false,
                                      static_cast<int64_t>(blockIdx.x) * COLS);
}

// The inverses of every diagonal block of a solve, in one launch: block
// b = blockIdx.y (order s_b ≤ LEAF at (off_b, off_b)) solves its transpose
// against the identity, so W_b = W + b·LEAF² (column-major, pitch LEAF)
// receives the transpose of its inverse: W_b[k·LEAF + i] = L_b⁻¹(k, i).
// The first launch of its solve: waits for the previous launch on the
// stream before anything else (the previous solve may still read W).
// COLS right-hand sides (columns of the identity) per thread block: block b
// = blockIdx.x, columns j0 = (gridDim.y − 1 − blockIdx.y)·COLS. A block
// with right-hand sides j0 .. j0+COLS-1 walks the groups up to the one
// holding j0+COLS-1 (the solutions are zero below the diagonal of Lᵀ's
// inverse), so the blocks of the last columns are the longest: they are
// launched first.
// sync (null: none): the synchronisation words of a chain launch that
// follows, zeroed by the first block once the previous launch is done.
template <int LEAF, int COLS>
__global__ void __launch_bounds__(LEAF, LEAF <= 256 ? 2 : 1)
    trsm_inverse_kernel(const uint16_t* __restrict__ A, int64_t lda, uint16_t* __restrict__ W,
                        const TriLeaves leaves, uint32_t* __restrict__ sync) {
  if (sync && blockIdx.x == 0 && blockIdx.y == 0) {
    grid_dependency_wait();
    for (int i = threadIdx.x; i < kChainSyncBytes / 4; i += blockDim.x) sync[i] = 0u;
  }
  const int b = blockIdx.x;
  const int s = static_cast<int>(leaves.size[b]);
  const int64_t j0 = static_cast<int64_t>(gridDim.y - 1 - blockIdx.y) * COLS;
  if (j0 >= s) {  // right-hand sides past the block's order: nothing to solve
    grid_dependency_wait();
    grid_launch_dependents();
    return;
  }
  trsm_leaf_body<COLS, LEAF>(A, lda, W + static_cast<int64_t>(b) * LEAF * LEAF, LEAF, leaves.off[b], 0, s, s, 0,
                             true, j0);
}

// X(:, j) = alpha · B(:, j) for the n × m column-major operands; FP16 in and
// out, FP32 product. In place when X == B (every element is read and written
// by the same thread). VEC: n, ldb, ldx multiples of 8 and both bases 16-byte
// aligned, 8 elements per 16-byte access.
template <bool VEC>
__global__ void scale_copy_kernel(const uint16_t* B, int64_t ldb, uint16_t* X, int64_t ldx,
                                  int64_t n, int64_t m, float alpha) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (VEC) {
    const int64_t per_col = n / 8, count = per_col * m;
    for (int64_t t = t0; t < count; t += stride) {
      const int64_t j = t / per_col, i = (t - j * per_col) * 8;
      if (!HG_DBG_INDEX(j, m) || !HG_DBG_INDEX(i + 7, n) || !HG_DBG_ALIGN(B + j * ldb + i, 16) ||
          !HG_DBG_ALIGN(X + j * ldx + i, 16))
        continue;
      uint4 v = *reinterpret_cast<const uint4*>(B + j * ldb + i);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
        const __half2 h = __floats2half2_rn(alpha * f.x, alpha * f.y);
        w[q] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(X + j * ldx + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    const int64_t count = n * m;
    for (int64_t t = t0; t < count; t += stride) {
      const int64_t j = t / n, i = t - j * n;
      const float v = __half2float(__ushort_as_half(B[j * ldb + i]));
      X[j * ldx + i] = __half_as_ushort(__float2half_rn(alpha * v));
    }
  }
}

// Resident blocks per SM of each width, measured once per device (0: not yet).
std::atomic<int> g_resident[kMaxDevices][3];

template <int COLS>
cudaError_t launch_width(const uint16_t* A, int64_t lda, uint16_t* X, int64_t ldx, int64_t off,
                         int s, int64_t m, int threads, bool chained, bool fwd, cudaStream_t stream) {
  const int64_t blocks = (m + COLS - 1) / COLS;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  PdlLaunch l(dim3(static_cast<unsigned>(blocks)), dim3(threads), leaf_smem<COLS>(), stream);
  return fwd ? cudaLaunchKernelEx(&l.cfg, trsm_leaf_kernel<COLS, true>, A, lda, X, ldx, off, s, m, chained ? 1 : 0)
             : cudaLaunchKernelEx(&l.cfg, trsm_leaf_kernel<COLS, false>, A, lda, X, ldx, off, s, m, chained ? 1 : 0);
}

// Sets both orientations' shared-memory size; the resident count is the same
// for both (same size, same launch bounds).
template <int COLS>
cudaError_t resident_blocks(int* out) {
  cudaError_t e = cudaFuncSetAttribute(trsm_leaf_kernel<COLS, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, leaf_smem<COLS>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(trsm_leaf_kernel<COLS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           leaf_smem<COLS>());
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, trsm_leaf_kernel<COLS, false>, kLeafMax,
                                                       leaf_smem<COLS>());
}

}  // namespace

cudaError_t launch_trsm_leaf(const uint16_t* A, int64_t lda, uint16_t* X, int64_t ldx, int64_t off,
                             int s, int64_t m, int num_sms, bool chained, bool fwd, cudaStream_t stream) {
  if (s < 1 || s > kLeafMax || m < 1 || num_sms < 1) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::atomic<int>* res = g_resident[dev];
  if (res[0] == 0) {
    int r8 = 0, r16 = 0, r32 = 0;
    if ((e = resident_blocks<8>(&r8)) != cudaSuccess || (e = resident_blocks<16>(&r16)) != cudaSuccess ||
        (e = resident_blocks<32>(&r32)) != cudaSuccess)
      return e;
    if (r8 < 1 || r16 < 1 || r32 < 1) return cudaErrorInvalidConfiguration;
    res[1] = r16;
    res[2] = r32;
    res[0] = r8;
  }
  // Width by estimated time: waves of blocks times the time of one block,
  // which is mostly the s barriers (≈ the same for every width) plus the
  // FMAs of its COLS right-hand sides.
  const int widths[3] = {8, 16, 32};
  int best = 0;
  double best_cost = 0.0;
  for (int w = 0; w < 3; ++w) {
    const int64_t blocks = (m + widths[w] - 1) / widths[w];
    const int64_t slots = static_cast<int64_t>(res[w]) * num_sms;
    const double cost = static_cast<double>((blocks + slots - 1) / slots) * (1.0 + widths[w] / 32.0);
    if (w == 0 || cost < best_cost) {
      best = w;
      best_cost = cost;
    }
  }
  const int threads = ((s + 31) / 32) * 32;
  switch (best) {
    case 0:
      return launch_width<8>(A, lda, X, ldx, off, s, m, threads, chained, fwd, stream);
    case 1:
      return launch_width<16>(A, lda, X, ldx, off, s, m, threads, chained, fwd, stream);
    default:
      return launch_width<32>(A, lda, X, ldx, off, s, m, threads, chained, fwd, stream);
  }
}

cudaError_t launch_trsm_inverse(const uint16_t* A, int64_t lda, uint16_t* W, const TriLeaves& leaves,
                                uint32_t* sync, cudaStream_t stream) {
  if (leaves.count < 1 || leaves.count > kMaxLeaves) return cudaErrorInvalidValue;
  for (int b = 0; b < leaves.count; ++b)
    if (leaves.size[b] < 1 || leaves.size[b] > kTrsmInverseLeaf) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  constexpr int LEAF = kTrsmInverseLeaf;
  static std::atomic<bool> attr_done[kMaxDevices];
  if (!attr_done[dev]) {
    if ((e = cudaFuncSetAttribute(trsm_inverse_kernel<LEAF, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  leaf_smem<16, LEAF>())) != cudaSuccess ||
        (e = cudaFuncSetAttribute(trsm_inverse_kernel<LEAF, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  leaf_smem<32, LEAF>())) != cudaSuccess ||
        (e = cudaFuncSetAttribute(trsm_inverse_kernel<LEAF, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  leaf_smem<64, LEAF>())) != cudaSuccess)
      return e;
    attr_done[dev] = true;
  }
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // Width by estimated time, one block per SM: a block of COLS right-hand
  // sides takes one group step per group up to its last column's, each step
  // ~(1.1 + COLS/40) µs (measured: 32 columns ~1.9 µs, 64 ~2.7 µs); blocks
  // are launched longest first, so the launch lasts about the longer of the
  // longest block and the total steps spread over the SMs.
  const int widths[3] = {16, 32, 64};
  int best = 1;
  double best_cost = 0.0;
  for (int w = 0; w < 3; ++w) {
    const int cols = widths[w];
    int64_t total = 0;
    int longest = 0;
    for (int b = 0; b < leaves.count; ++b) {
      const int groups = static_cast<int>((leaves.size[b] + 31) / 32);
      for (int64_t j0 = 0; j0 < leaves.size[b]; j0 += cols) {
        const int64_t last = (j0 + cols - 1) / 32;
        const int steps = static_cast<int>(last < groups - 1 ? last : groups - 1) + 1;
        total += steps;
        longest = steps > longest ? steps : longest;
      }
    }
    const int64_t spread = (total + sms - 1) / sms;
    const double cost = static_cast<double>(spread > longest ? spread : longest) * (1.1 + cols / 40.0);
    if (w == 0 || cost < best_cost) {
      best = w;
      best_cost = cost;
    }
  }
  const dim3 grid(static_cast<unsigned>(leaves.count), static_cast<unsigned>(LEAF / widths[best]));
  switch (best) {
    case 0: {
      PdlLaunch l(grid, dim3(LEAF), leaf_smem<16, LEAF>(), stream);
      return cudaLaunchKernelEx(&l.cfg, trsm_inverse_kernel<LEAF, 16>, A, lda, W, leaves, sync);
    }
    case 1: {
      PdlLaunch l(grid, dim3(LEAF), leaf_smem<32, LEAF>(), stream);
      return cudaLaunchKernelEx(&l.cfg, trsm_inverse_kernel<LEAF, 32>, A, lda, W, leaves, sync);
    }
    default: {
      PdlLaunch l(grid, dim3(LEAF), leaf_smem<64, LEAF>(), stream);
      return cudaLaunchKernelEx(&l.cfg, trsm_inverse_kernel<LEAF, 64>, A, lda, W, leaves, sync);
    }
  }
}

cudaError_t launch_scale_copy(const uint16_t* B, int64_t ldb, uint16_t* X, int64_t ldx, int64_t n,
                              int64_t m, float alpha, int num_sms, cudaStream_t stream) {
  const bool vec = n % 8 == 0 && ldb % 8 == 0 && ldx % 8 == 0 &&
                   ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(X)) & 15u) == 0;
  const int64_t count = vec ? n / 8 * m : n * m;
  int64_t blocks = (count + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  PdlLaunch l(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream);
  return cudaLaunchKernelEx(&l.cfg, vec ? scale_copy_kernel<true> : scale_copy_kernel<false>, B, ldb, X, ldx,
                            n, m, alpha);
}

// The -DHGEMM_DEBUG build's check word of this file (null otherwise).
HG_DEBUG_WORD_ACCESSOR(trsm)

}  // namespace hg
