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
cudaError_t launch_tc_128x64(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
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
// Bytes of the workspace's synchronisation words of the one-launch solve.
constexpr int kChainSyncBytes = 4096;
// sync (may be null): kChainSyncBytes that the launch zeroes (after waiting
// for the previous launch on the stream) for a chain launch that follows.
cudaError_t launch_trsm_inverse(const uint16_t* A, int64_t lda, uint16_t* W, const TriLeaves& leaves,
                                uint32_t* sync, cudaStream_t stream);
// fwd: the literal orientation A·X = alpha·B (forward substitution).
cudaError_t launch_trsm_leaf(const uint16_t* A, int64_t lda, uint16_t* X, int64_t ldx, int64_t off,
                             int s, int64_t m, int num_sms, bool chained, bool fwd, cudaStream_t stream);


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
constexpr int kNarrowBN = 64;  // single-CTA kernel for outputs of one wave of 128×64 tiles
constexpr int kTcBK = 64;
constexpr int kPairBN = 256;   // pair kernel: 256×256 tiles, 128 B rows per CTA
constexpr int kPairRingBytes = 6 * 32768;  // pair kernel: six whole-tile stages of A and B
constexpr int kEpiRows = 32;   // rows of one staged C box (one epilogue warp)
constexpr int kEpiCols = 64;   // columns of one staged C box (128 bytes)

}  // namespace hg
