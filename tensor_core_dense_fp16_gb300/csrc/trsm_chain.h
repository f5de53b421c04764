// trsm_chain.h — host-side interface of the one-launch triangular solve
// (hgemm_trsm_chain.cu), shared with the C-ABI layer (hgemm_api.cu). Not
// part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace hg {

// The solve with inverses as one persistent, cooperative launch (see
// hgemm_trsm_chain.cu): one phase per diagonal block in the order of the
// solve, grid-wide barriers between phases. Xᵀ is the m × n row-major view
// of X (column j of X is row j). A phase is a list of tile groups:
//   product   Xᵀ_k := Xᵀ_k · L_k⁻¹ (· L_k⁻ᵀ for A·X = B) − Xᵀ_{k−1} · M_k,
//             a K segment per term (the second absent for the first block);
//   coupling  M_{k+1} := −C(k, k+1) · L_{k+1}⁻¹ into a free workspace slot,
//             C(k, k+1) the triangle's block coupling block k to block k+1;
//   update    Xᵀ_c −= Xᵀ_{k−1} · C(k−1, c) for every block c after k,
// and, only where X := alpha·B cannot be folded into the first phases, a
// copy phase first.
enum ChainKind : int { kChainCopy = 0, kChainProduct = 1, kChainUpdate = 2, kChainCoupling = 3 };
enum ChainMap : int { kChainMapX = 0, kChainMapB = 1, kChainMapW = 2, kChainMapWRagged = 3, kChainMapA = 4 };
constexpr int kChainMaxLeaves = 16;
constexpr int kChainMaxGroups = 1 + 3 * kChainMaxLeaves;
// Words of the workspace's synchronisation area (zeroed by the inverses'
// launch before the chain starts): the grid barrier's arrival count, the
// launch's abort flag, then one counter per 64 rows of Xᵀ.
constexpr int kChainSyncBarrier = 0;
constexpr int kChainSyncAbort = 1;
constexpr int kChainSyncRowGroup0 = 32;
constexpr int kChainMaxRowGroups = kChainSyncBytes / 4 - kChainSyncRowGroup0;

// One group of tiles: bm × bn (bm 64 or 128, bn 64, 128 or 256) over output
// rows [0, rows) and columns [n0, n_end). First K segment: ksteps steps of
// 64, the first operand at (k, row) = (a_kbase + 64·kk, a_mbase + row) in
// map a_map (M-contiguous when a_mn), the second at (k, n) = (b_kbase +
// 64·kk, b_nbase + column − n0) in map b_map (N-contiguous when b_mn).
// Second segment (products, ksteps2 > 0): Xᵀ columns a2_kbase + 64·kk with
// the W map's rows b2_kbase + 64·kk, N-contiguous. Products store scale ·
// acc to X, couplings scale · acc to W slot out_slot (rows of 512), updates
// the previous value (alpha·B when old_from_b) minus acc. Critical
// products: every 64-row group of Xᵀ has a counter that each tile covering it
// raises once its Xᵀ boxes have landed; a tile stores its rows only when
// the counter has reached rg_target (the tiles of one row range read each
// other's columns).
struct ChainGroup {
  uint32_t flags;  // see chain_group_flags
  int rows, n0, n_end;
  int a_kbase, a_mbase, ksteps;
  int b_kbase, b_nbase;
  int a2_kbase, b2_kbase, ksteps2;
  int out_slot;
  float scale;
  uint32_t rg_target;
};
// last: the phase's last group; critical: the phase's products, on CTAs of their own
__host__ __device__ constexpr uint32_t chain_group_flags(int kind, int a_map, int a_mn, int b_map, int b_mn, int bm,
                                                         int bn, int old_from_b, int last, int critical) {
  return static_cast<uint32_t>(kind | (a_map << 2) | (a_mn << 5) | (b_map << 6) | (b_mn << 9) | ((bm / 64) << 10) |
                               ((bn / 64) << 12) | (old_from_b << 15) | (last << 16) | (critical << 17));
}

struct ChainArgs {
  uint16_t* X;
  int64_t ldx;
  const uint16_t* B;  // the right-hand side, may be X
  int64_t ldb;
  uint16_t* W;        // the workspace's slots of 512 × 512 (couplings are written here)
  float alpha;
  int m, n;
  int copy_vec;       // the copy phase moves 8 elements per access
  uint32_t* sync;     // kChainSyncBytes in the workspace
  int* status;
  unsigned long long timeout_ns;
  int inject;
  int num_groups;
  ChainGroup group[kChainMaxGroups];
};

// x: Xᵀ (m × n, pitch ldx); b: Bᵀ (pitch ldb), or a copy of x; w: the
// workspace's slots (count·512 rows of 512); wr: the ragged last block's
// inverse (s × s, pitch 512), or a copy of w; a: the triangle as stored (n
// columns of n rows, pitch lda). Every map has 64 × 64 boxes with 128-byte
// swizzling.
cudaError_t launch_trsm_chain(const CUtensorMap& x, const CUtensorMap& b, const CUtensorMap& w,
                              const CUtensorMap& wr, const CUtensorMap& a, const ChainArgs& args, int grid,
                              cudaStream_t stream);
// Largest grid of the chain kernel that is co-resident on this device (0 on error).
int chain_max_grid(int num_sms);

}  // namespace hg
