// internal.h — host-side interface between the C-ABI layer (hgemm_api.cu)
// and the kernel translation units. Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace hg {

// Watchdog codes written to the device status word by a wait that gave up.
enum WatchdogCode : int {
  kWdNone = 0,
  kWdProducerEmpty = 1,   // TMA producer waiting for a free smem stage
  kWdMmaFull = 2,         // MMA issuer waiting for a loaded smem stage
  kWdMmaAccEmpty = 3,     // MMA issuer waiting for the epilogue to free TMEM
  kWdEpiAccFull = 4,      // epilogue waiting for a finished accumulator
  kWdDrain = 5,           // end-of-kernel drain of in-flight copies or MMAs
  kWdReduce = 6,          // split-K owner waiting for the other slices' partials
  kWdGridBarrier = 7,     // a CTA of a cooperative launch waiting for all others at a phase boundary
  kWdRowGroup = 8,        // an epilogue waiting for the CTAs that read the rows it overwrites
};

// The fused epilogue ("GPU架构与CUDA", 核函数融合): each FP32 accumulator
// becomes alpha·acc + beta·C_old + bias[col], then max(·, 0) when relu is
// set, before the single rounding to FP16. mode 0: plain product (the
// accumulator is stored as is); 1: fused, C not read; 2: fused, C read.
struct EpiArgs {
  float alpha, beta;
  const uint16_t* bias;  // N FP16 values (one per column of C), or null
  int relu;
  int mode;
};

// Everything a tensor-core launch needs besides the tensor maps.
struct TcArgs {
  int M, N, K;
  int num_m, num_n, num_kb;  // tiles along M and N, 64-wide K blocks
  int num_tiles;             // work units: whole tiles, then tile parts
  int full_tiles;            // units below this index are whole tiles; the rest are
                             // parts of part_cols columns of the last tiles (pair kernel)
  int part_cols;             // 128 or 64
  int stages, stage_bytes;   // operand ring geometry (pair kernel)
  int group_m;               // rasterisation group height (in M tiles)
  int grid;                  // persistent CTAs
  int* status;               // device watchdog word
  unsigned long long timeout_ns;
  int inject;                // HGEMM_INJECT_* (testing the watchdog)
  EpiArgs epi;
  const uint16_t* C;         // C itself, read in epilogue mode 2
  int64_t ldc;               // C's row pitch in elements
  int a_mn, b_mn;            // pair kernel: A stored M-contiguous (K×M), B stored
                             // N-contiguous (K×N); else K-contiguous
  int batch_tiles;           // pair kernel: whole tiles per product of a batch of
                             // equal products in one launch (0: a single product)
  int batch_shift;           // product j of the batch is the first one with A's K,
                             // B's N and K, and C's N coordinates shifted by j·batch_shift
};

// Plain-pointer launch arguments for the kernels that do not use TMA.
struct PlainArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* C;
  int64_t M, N, K;
  int64_t lda, ldb, ldc;     // row pitches in elements
  int* status;
  unsigned long long timeout_ns;
  EpiArgs epi;
  int a_mn = 0, b_mn = 0;    // A(i,k) at A[k*lda + i]; B(k,j) at B[k*ldb + j]
};

// The diagonal blocks ("leaves") of a triangular product, for one batched
// launch of masked products.
constexpr int kMaxLeaves = 128;
struct TriLeaves {
  int count;
  int64_t off[kMaxLeaves];   // first row (and column) of each block in the triangle
  int64_t size[kMaxLeaves];  // its order
};

// Every kernel here is launched with programmatic stream serialization: it
// may start while the previous kernel on the stream is still running, and
// waits for it (griddepcontrol.wait) before touching memory that kernel may
// write, so its launch and prologue overlap the previous kernel's tail.
struct PdlLaunch {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg;
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) : attr{}, cfg{} {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // clusters of x CTAs set at launch time
  void cluster(unsigned x) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
};

// Launchers (each enqueues one kernel on `stream` and returns the launch
// error, if any). Shared-memory attributes are set on first use per device.
cudaError_t launch_tc_128x256(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                              const TcArgs& args, cudaStream_t stream);
// b_part: the B map with part_cols / 2-row boxes, for the tile parts of the last wave.
cudaError_t launch_tc_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b_part,
                           const CUtensorMap& c, const TcArgs& args, cudaStream_t stream);
// Largest number of co-resident 2-CTA clusters of the pair kernel.
int pair_max_clusters(int num_sms);
// Wide pair kernel: 256×512 tiles per CTA pair.
cudaError_t launch_tc_wide(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const TcArgs& args, cudaStream_t stream);
int wide_max_clusters(int num_sms);
// Split-K cluster kernel for few output tiles: `split` K-slices, one cluster
// of 2*split CTAs per 256×tile_n tile (args.num_tiles of them); tile_n 256
// with 2, 3 or 4 slices, or tile_n 128 with 2.
cudaError_t launch_skinny(int split, int tile_n, const CUtensorMap& a, const CUtensorMap& b,
                          const CUtensorMap& c, const TcArgs& args, cudaStream_t stream);
// Largest number of co-resident clusters of the split-K kernel.
int skinny_max_clusters(int split, int tile_n, int num_sms);
// K = 0: C := f(beta·C_old + bias) elementwise (plain mode: +0).
cudaError_t launch_empty_sum(uint16_t* C, int64_t M, int64_t N, int64_t ldc, const EpiArgs& epi,
                             cudaStream_t stream);
cudaError_t launch_generic(const PlainArgs& args, int num_sms, cudaStream_t stream);
// A kernel that does nothing: one CTA of one warp, or (pair_config) one CTA
// per SM in clusters of two with `smem_bytes` of dynamic shared memory each.
cudaError_t launch_floor(int pair_config, int num_sms, int smem_bytes, cudaStream_t stream);
// Dynamic shared memory of one pair-kernel CTA.
int pair_smem_bytes();
// Every leaf b: C + off = (A operand + off) · lower(B operand at (off, off)),
// M × size (see hgemm_generic.cu).
cudaError_t launch_tri_leaves(const PlainArgs& args, const TriLeaves& leaves, int num_sms,
                              cudaStream_t stream);
// The same on the tensor cores for leaves whose orders are multiples of 64
// (see hgemm_trileaf.cu): x maps Bᵀ (m × n, 128×64 boxes), l maps the rows
// of the triangle (column i of A as row i, n × n, 64×64 boxes), c maps Cᵀ
// (m × n, 32×64 boxes); args.num_m row tiles of 128 per leaf.
// ext[b]: K columns past leaf b's own block that its product also covers,
// [off_b + s_b, off_b + s_b + ext[b]) (whole rows of the second operand:
// the off-diagonal updates of the blocks whose first half holds leaf b), a
// multiple of 64, or 0.
struct TriLeafExt {
  int32_t ext[kMaxLeaves];
};
cudaError_t launch_tri_leaves_tc(const CUtensorMap& x, const CUtensorMap& l, const CUtensorMap& c,
                                 const TcArgs& args, const TriLeaves& leaves, const TriLeafExt& ext,
                                 cudaStream_t stream);

// Triangular solve Aᵀ·X = alpha·B (see hgemm_trsm.cu): the largest diagonal
// block solved by substitution; X(:, j) = alpha·B(:, j) over n × m
// column-major operands (X == B allowed); the solve of the diagonal block of
// order s at (off, off) for all m right-hand sides, in place in X.
constexpr int kTrsmLeaf = 256;
cudaError_t launch_scale_copy(const uint16_t* B, int64_t ldb, uint16_t* X, int64_t ldx, int64_t n,
                              int64_t m, float alpha, int num_sms, cudaStream_t stream);
// chained: an earlier launch of the same solve precedes this one on the
// stream (the kernel may then read A before waiting for it).
// The inverses of every diagonal block (leaf b of order s_b ≤ kTrsmInverseLeaf
// at (off_b, off_b)) in one launch: W + b·kTrsmInverseLeaf² receives,
// column-major with pitch kTrsmInverseLeaf, the transpose of the block's
// inverse (row k of the inverse is contiguous), FP16.
constexpr int kTrsmInverseLeaf = 512;
// sync (may be null): kChainSyncBytes that the launch zeroes (after waiting
// for the previous launch on the stream) for a chain launch that follows.
cudaError_t launch_trsm_inverse(const uint16_t* A, int64_t lda, uint16_t* W, const TriLeaves& leaves,
                                uint32_t* sync, cudaStream_t stream);
// fwd: the literal orientation A·X = alpha·B (forward substitution).
cudaError_t launch_trsm_leaf(const uint16_t* A, int64_t lda, uint16_t* X, int64_t ldx, int64_t off,
                             int s, int64_t m, int num_sms, bool chained, bool fwd, cudaStream_t stream);

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
constexpr int kChainSyncBytes = 4096;
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

// Address of the device watchdog word on the current device.
cudaError_t status_word_address(int** addr);

// The -DHGEMM_DEBUG build's check words, one per kernel file (each sets
// *out to null in the release build).
cudaError_t debug_word_tc(int** out);
cudaError_t debug_word_tc2(int** out);
cudaError_t debug_word_tc2w(int** out);
cudaError_t debug_word_skinny(int** out);
cudaError_t debug_word_generic(int** out);
cudaError_t debug_word_trsm(int** out);
cudaError_t debug_word_trileaf(int** out);
cudaError_t debug_word_chain(int** out);
constexpr int kDebugWords = 8;

// Co-residency limits of the cluster kernels on one device, measured once
// (or nominal GB300 figures when no device has been queried).
struct DeviceProfile {
  int num_sms;
  int pair_clusters;    // co-resident 2-CTA clusters of the pair kernel
  int split2_clusters;  // co-resident 4-CTA clusters of the split-K kernel
  int split3_clusters;  // co-resident 6-CTA clusters
  int split4_clusters;  // co-resident 8-CTA clusters
  int split2n_clusters;  // co-resident 4-CTA clusters of the 128-column split-K kernel
};

// Kernel choice for a TMA-able product. Returns an HGEMM_PATH_* value and,
// for the split-K path, the number of K-slices in *split and the tile width
// in *tile_n. forced: a forced HGEMM_PATH_* or -1; forced_split and
// forced_tile_n: a forced split-K configuration or 0; fused: the product
// has a fused epilogue (hgemm_ex other than the plain product).
int choose_tma_path(int64_t M, int64_t N, int64_t K, const DeviceProfile& dev, int forced,
                    int forced_split, int forced_tile_n, bool fused, int* split, int* tile_n);

// Tile geometry of the tensor-core path, for the host-side tensor maps.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
constexpr int kPairBN = 256;   // pair kernel: 256×256 tiles, 128 B rows per CTA
constexpr int kPairRingBytes = 6 * 32768;  // pair kernel: six whole-tile stages of A and B
constexpr int kEpiRows = 32;   // rows of one staged C box (one epilogue warp)
constexpr int kEpiCols = 64;   // columns of one staged C box (128 bytes)

}  // namespace hg
