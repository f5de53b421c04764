// hgemm_api.cu — the C ABI declared in include/hgemm.h: argument checks,
// path selection, TMA tensor-map encoding and kernel dispatch.
//
// The entry point follows the launcher of "Nvidia Tensor Core-MMA PTX编程入门",
// §4 示例 (pointers to A, B, C and the sizes M, N, K; the launcher picks the
// grid) and adds the caller's stream ("GPU架构与CUDA", 流与并发). The library
// never allocates device memory: buffers come from the caller, who owns them
// ("GPU架构与CUDA", 内存池分配器: allocation belongs to a caching allocator
// such as PyTorch's, not to every call).
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <vector>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "hgemm.h"
#include "debug.cuh"
#include "internal.h"
#include "trsm_chain.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int64_t kTrmmLeaf = 256;  // diagonal blocks of at most this order are leaves
// Updates of at most this many multiply-adds (m·s1·s2; 8192 × 1024 × 1024)
// are carried by the tensor-core leaves. Measured: at n = m = 8192 carrying
// the updates of blocks up to 1024, 2048 and 4096 gave 407, 397 and 400 µs
// (the 8192 × 2048 × 2048 updates run better on the pair kernel); at
// n = 4096, m = 256 (every update small) 42.5, 37.9 and 34.5 µs.
constexpr int64_t kTrmmFoldMacs = int64_t(1) << 33;

thread_local int t_last_cuda_error = 0;
std::atomic<int> g_forced_path{-1};
std::atomic<int> g_forced_split{0};  // split * 1024 + tile_n, or 0
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_inject{HGEMM_INJECT_NONE};
std::atomic<int> g_trsm_schedule{HGEMM_TRSM_AUTO};  // hgemm_force_trsm_schedule
thread_local int t_trsm_schedule = 0;               // hgemm_trsm_last_schedule

struct DeviceState {
  std::atomic<int> ready{0};  // 0 unknown, 1 supported, -1 unsupported
  int id = 0;
  int num_sms = 0;
  hg::DeviceProfile prof{};
};
DeviceState g_devices[kMaxDevices];

// Device addresses of the library's static device variables (the watchdog
// word, the fixed TRSM workspace) belong to the context they were looked up
// in. Each host thread keeps the ones of its current context and looks them
// up again when that context changes (another context on the device, or the
// primary context recreated after a device reset).
struct ContextCache {
  unsigned long long ctx = 0;  // cuCtxGetId of the context, 0: none cached
  int* status = nullptr;       // the watchdog word
  void* noalloc = nullptr;     // hgemm_trsm_noalloc's array (null: not yet looked up)
  int* debug[hg::kDebugWords] = {};  // the debug build's check words (null in the release build)
};
thread_local ContextCache t_ctx;
thread_local int t_debug_code = 0;  // the last check code hgemm_device_status read

// The debug build's check words in the current context.
cudaError_t debug_words(int* (&out)[hg::kDebugWords]) {
  cudaError_t (*const get[hg::kDebugWords])(int**) = {hg::debug_word_tc,      hg::debug_word_tc2,
                                                      hg::debug_word_tc2w,    hg::debug_word_skinny,
                                                      hg::debug_word_generic, hg::debug_word_trsm,
                                                      hg::debug_word_trileaf, hg::debug_word_chain};
  for (int i = 0; i < hg::kDebugWords; ++i) {
    const cudaError_t e = get[i](&out[i]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Unique identity (for the life of the process) of the calling thread's
// current context, or 0 when it cannot be determined.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// One product: operands, sizes and row pitches in elements (A(i,k) at
// A[i*lda + k], B(k,j) at B[j*ldb + k], C(i,j) at C[i*ldc + j]; with a_mn,
// A(i,k) at A[k*lda + i]; with b_mn, B(k,j) at B[k*ldb + j]).
struct Gemm {
  const void* A;
  const void* B;
  void* C;
  int64_t M, N, K;
  int64_t lda, ldb, ldc;
  bool a_mn = false, b_mn = false;
  // where a fused epilogue reads C_old (row pitch ld_src), when not from C
  // itself: the TMA paths only (the generic kernel reads C_old from C)
  const void* c_src = nullptr;
  int64_t ld_src = 0;
};

Gemm dense(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K) {
  return Gemm{A, B, C, M, N, K, K, K, N};
}
std::mutex g_device_mu;

// GB300 figures, used by hgemm_select_path before any device has been used
// in this process: 152 SMs; co-resident clusters of 2, 4, 6 and 8 CTAs of
// ~200-225 KB of shared memory each, as cudaOccupancyMaxActiveClusters
// reports them on this part.
constexpr hg::DeviceProfile kNominalProfile{152, 76, 36, 23, 15, 36};
std::atomic<const hg::DeviceProfile*> g_last_profile{&kNominalProfile};

// The plain product: the accumulator is stored as it is.
constexpr hg::EpiArgs kPlainEpilogue{1.0f, 0.0f, nullptr, 0, 0};

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return HGEMM_ERR_CUDA;
}

// Checks the current device once: compute capability 10.3 and the watchdog
// word's address. Returns HGEMM_OK and the state, or an error status.
int current_device(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return HGEMM_ERR_UNSUPPORTED_DEVICE;
  // The tensor maps are encoded by a driver-API call, which needs the
  // device's context current on this host thread: a thread whose runtime
  // calls so far needed no context (streams and memory from a caching
  // allocator, say) may not have it yet. Bind it once per thread and device.
  thread_local int t_bound_device = -1;
  if (t_bound_device != dev) {
    if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e);
    t_bound_device = dev;
  }
  DeviceState& st = g_devices[dev];
  int r = st.ready.load(std::memory_order_acquire);
  if (r == 0) {
    std::lock_guard<std::mutex> lock(g_device_mu);
    r = st.ready.load(std::memory_order_relaxed);
    if (r == 0) {
      int major = 0, minor = 0, sms = 0;
      if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e);
      if (major != 10 || minor != 3) {
        r = -1;
      } else {
        st.id = dev;
        st.num_sms = sms;
        st.prof.num_sms = sms;
        st.prof.pair_clusters = hg::pair_max_clusters(sms);
        st.prof.split2_clusters = hg::skinny_max_clusters(2, 256, sms);
        st.prof.split3_clusters = hg::skinny_max_clusters(3, 256, sms);
        st.prof.split4_clusters = hg::skinny_max_clusters(4, 256, sms);
        st.prof.split2n_clusters = hg::skinny_max_clusters(2, 128, sms);
        r = 1;
      }
      st.ready.store(r, std::memory_order_release);
    }
  }
  if (r < 0) return HGEMM_ERR_UNSUPPORTED_DEVICE;
  // the watchdog word's address in the calling thread's current context
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || ctx != t_ctx.ctx) {
    int* status = nullptr;
    if ((e = hg::status_word_address(&status)) != cudaSuccess) return cuda_fail(e);
    ContextCache fresh{ctx, status, nullptr, {}};
    if ((e = debug_words(fresh.debug)) != cudaSuccess) return cuda_fail(e);
    t_ctx = fresh;
  }
  g_last_profile.store(&st.prof, std::memory_order_release);
  *out = &st;
  return HGEMM_OK;
}

bool ranges_overlap(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  if (!a || !b || abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Host-only argument checks shared by every entry point.
int validate(const Gemm& g) {
  const int64_t M = g.M, N = g.N, K = g.K;
  if (M < 0 || N < 0 || K < 0 || M > HGEMM_MAX_DIM || N > HGEMM_MAX_DIM || K > HGEMM_MAX_DIM)
    return HGEMM_ERR_INVALID_ARG;
  // pitches cover a stored row and stay far from overflow
  const int64_t ld_lim = int64_t(1) << 40;
  const int64_t a_cols = g.a_mn ? M : K, a_rows = g.a_mn ? K : M;
  const int64_t b_cols = g.b_mn ? N : K, b_rows = g.b_mn ? K : N;
  if (g.lda < a_cols || g.ldb < b_cols || g.ldc < N || g.lda > ld_lim || g.ldb > ld_lim ||
      g.ldc > ld_lim)
    return HGEMM_ERR_INVALID_ARG;
  // element spans (each < 2^61) and byte spans (< 2^62) cannot overflow
  using u128 = unsigned __int128;
  auto span = [](int64_t rows, int64_t ld, int64_t cols) -> u128 {
    return (rows > 0 && cols > 0) ? static_cast<u128>(rows - 1) * ld + cols : 0;
  };
  const u128 sa = span(a_rows, g.lda, a_cols), sb = span(b_rows, g.ldb, b_cols), sc = span(M, g.ldc, N);
  const u128 lim = static_cast<u128>(1) << 61;
  if (sa >= lim || sb >= lim || sc >= lim) return HGEMM_ERR_INVALID_ARG;
  if ((sa && !g.A) || (sb && !g.B) || (sc && !g.C)) return HGEMM_ERR_INVALID_ARG;
  // FP16 elements: every pointer must be at least 2-byte aligned
  if ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.B) |
       reinterpret_cast<uintptr_t>(g.C)) & 1u)
    return HGEMM_ERR_INVALID_ARG;
  // C is written while A and B are read: their spans must not meet
  if (sc && (ranges_overlap(g.C, 2 * static_cast<uint64_t>(sc), g.A, 2 * static_cast<uint64_t>(sa)) ||
             ranges_overlap(g.C, 2 * static_cast<uint64_t>(sc), g.B, 2 * static_cast<uint64_t>(sb))))
    return HGEMM_ERR_ALIAS;
  return HGEMM_OK;
}

// TMA needs 16-byte-aligned bases and row pitches; the epilogue's 16-byte
// reads of C need N to be a multiple of 8 as well.
bool tma_ok(const Gemm& g) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return al16(g.A) && al16(g.B) && al16(g.C) && g.lda % 8 == 0 && g.ldb % 8 == 0 &&
         g.ldc % 8 == 0 && g.N % 8 == 0 && (!g.c_src || (al16(g.c_src) && g.ld_src % 8 == 0));
}

int choose_path(const Gemm& g, const hg::DeviceProfile& prof, bool fused, int* split, int* tile_n) {
  *split = 1;
  *tile_n = hg::kPairBN;
  const int64_t M = g.M, N = g.N, K = g.K;
  if (M == 0 || N == 0) return HGEMM_PATH_NONE;
  if (K == 0) return HGEMM_PATH_ZERO;
  const bool tma = tma_ok(g);
  const int forced = g_forced_path.load(std::memory_order_relaxed);
  if (forced == HGEMM_PATH_GENERIC || !tma) return HGEMM_PATH_GENERIC;
  const int fs = g_forced_split.load(std::memory_order_relaxed);
  const int path = hg::choose_tma_path(M, N, K, prof, forced, fs >> 10, fs & 1023, fused, split, tile_n);
  // M- or N-contiguous operands: the wide, pair and split-K kernels read
  // them as MN-major tiles; the single-CTA kernel takes K-major ones only
  if ((g.a_mn || g.b_mn) && (path == HGEMM_PATH_TC || path == HGEMM_PATH_TC_NARROW))
    return HGEMM_PATH_TC_PAIR;
  return path;
}

}  // namespace

namespace hg {

int choose_tma_path(int64_t M, int64_t N, int64_t K, const DeviceProfile& dev, int forced,
                    int forced_split, int forced_tile_n, bool fused, int* split, int* tile_n) {
  *split = 1;
  *tile_n = kPairBN;
  const int64_t num_m = (M + 2 * kTcBM - 1) / (2 * kTcBM);
  const int64_t num_kb = (K + kTcBK - 1) / kTcBK;
  // Split-K configurations: S K-slices over 256-column tiles (S = 2, 3, 4)
  // or 2 slices over 128-column tiles, one cluster of 2·S CTAs per tile.
  // A configuration is usable when all its clusters fit on the device at
  // once and every slice has a K block; `need_idle` also requires that the
  // unsplit pair kernel would leave at least half of the SM pairs idle and
  // that the split asks for no more pairs than the device has.
  auto usable = [&](int s, int bn, bool need_idle) {
    const int64_t tiles = num_m * ((N + bn - 1) / bn);
    const int fits = bn == 128 ? (s == 2 ? dev.split2n_clusters : 0)
                               : (s == 2 ? dev.split2_clusters
                                  : s == 3 ? dev.split3_clusters
                                  : s == 4 ? dev.split4_clusters : 0);
    if (num_kb < s || tiles > fits) return false;
    if (need_idle && (2 * num_m * ((N + kPairBN - 1) / kPairBN) > dev.pair_clusters ||
                      s * tiles > dev.pair_clusters))
      return false;
    return true;
  };
  // Cost estimate in microseconds: each SM takes in its slice's operands at
  // ~112 GB/s (measured cap of one SM's intake), and sends and receives its
  // share of the FP32 partial sums at an effective ~21 GB/s (fitted to the
  // measured launches of 4096×256×4096 in both tile widths).
  auto cost = [&](int s, int bn) {
    const double intake = static_cast<double>(num_kb) / s * (kTcBM + bn / 2) * kTcBK * 2;
    const double exchange = static_cast<double>(kTcBM) * bn * 4 * (s - 1) / s;
    return intake / 112e3 + exchange / 21e3;
  };
  auto choose = [&](bool need_idle) -> bool {
    if (forced_split > 0 && usable(forced_split, forced_tile_n, false)) {
      *split = forced_split;
      *tile_n = forced_tile_n;
      return true;
    }
    const int cand[4][2] = {{2, 128}, {4, 256}, {3, 256}, {2, 256}};
    double best = 0;
    bool found = false;
    for (const auto& c : cand) {
      if (!usable(c[0], c[1], need_idle)) continue;
      const double t = cost(c[0], c[1]);
      if (!found || t < best) {
        best = t;
        *split = c[0];
        *tile_n = c[1];
        found = true;
      }
    }
    return found;
  };
  if (forced == HGEMM_PATH_TC || forced == HGEMM_PATH_TC_NARROW || forced == HGEMM_PATH_TC_PAIR ||
      forced == HGEMM_PATH_TC_WIDE)
    return forced;
  if (forced == HGEMM_PATH_SKINNY) return choose(false) ? HGEMM_PATH_SKINNY : HGEMM_PATH_TC_PAIR;
  // Exchanging the partial sums costs a few microseconds; splitting pays
  // when each pair would otherwise walk a long K (48 blocks or more).
  if (num_kb >= 48 && choose(true)) return HGEMM_PATH_SKINNY;
  // An output that one wave of 128×64 tiles covers: one CTA per tile, no
  // cluster. With a short K the launch is bound by its fixed chain of
  // dependent steps, which the single-CTA kernel keeps shorter than the
  // pair kernel's (measured, flushed: 256³ 8.2 against 8.9 µs, 1000³ 12.3
  // against 14.3 µs), though each CTA reads 20% more operand bytes than in
  // the pair kernel's 64-column parts.
  const int64_t narrow_tiles = ((M + kTcBM - 1) / kTcBM) * ((N + kNarrowBN - 1) / kNarrowBN);
  if (narrow_tiles <= dev.num_sms) return HGEMM_PATH_TC_NARROW;
  // A CTA pair covers 256 rows; with 128 rows or fewer half of it would idle.
  if (M <= kTcBM) return HGEMM_PATH_TC;
  // 256×512 tiles move 25% fewer operand bytes per flop than 256×256 ones
  // (measured in runs of 300 launches at 8192³: +1.5%, less power for the
  // same work under the power cap); take them when there are enough of them
  // to give every pair a tile. Their accumulator fills TMEM, so the tensor
  // cores wait for each epilogue: with a fused epilogue the 256×256 tiles,
  // whose accumulators are double-buffered, are faster (~8% at 8192³).
  const int64_t wide_tiles = ((M + 2 * kTcBM - 1) / (2 * kTcBM)) * ((N + 2 * kPairBN - 1) / (2 * kPairBN));
  if (!fused && wide_tiles >= dev.pair_clusters) return HGEMM_PATH_TC_WIDE;
  return HGEMM_PATH_TC_PAIR;
}

}  // namespace hg

namespace {

bool tail_split_setting() {
  static const bool v = [] {
    const char* e = std::getenv("HGEMM_TAIL_SPLIT");
    return !(e && e[0] == '0');
  }();
  return v;
}

int group_m_setting() {
  static const int v = [] {
    const char* e = std::getenv("HGEMM_GROUP_M");
    const int x = e ? std::atoi(e) : 0;
    return x > 0 ? x : 12;
  }();
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major FP16 matrix [rows][cols] with rows `pitch`
// elements apart, read or written in boxes of box_rows × box_cols
// (box_cols * 2 == 128 bytes: one swizzle row).
int encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t pitch,
               int box_rows, int box_cols) {
  auto encode = tensor_map_encoder();
  if (!encode) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                      strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return HGEMM_OK;
}

// bn: the tile width, hg::kTcBN (128×256 tiles) or hg::kNarrowBN (128×64).
int run_tc(const Gemm& g, const hg::EpiArgs& epi, const DeviceState& dev, cudaStream_t stream,
           int bn) {
  const void* A = g.A;
  const void* B = g.B;
  void* C = g.C;
  const int64_t M = g.M, N = g.N, K = g.K;
  CUtensorMap ma, mb, mc;
  int rc;
  if ((rc = encode_map(&ma, A, M, K, g.lda, hg::kTcBM, hg::kTcBK)) != HGEMM_OK) return rc;
  if ((rc = encode_map(&mb, B, N, K, g.ldb, bn, hg::kTcBK)) != HGEMM_OK) return rc;
  if ((rc = encode_map(&mc, C, M, N, g.ldc, hg::kEpiRows, hg::kEpiCols)) != HGEMM_OK) return rc;
  hg::TcArgs args{};
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.K = static_cast<int>(K);
  args.num_m = static_cast<int>((M + hg::kTcBM - 1) / hg::kTcBM);
  args.num_n = static_cast<int>((N + bn - 1) / bn);
  args.num_kb = static_cast<int>((K + hg::kTcBK - 1) / hg::kTcBK);
  const int64_t tiles = static_cast<int64_t>(args.num_m) * args.num_n;
  if (tiles > 0x7FFFFFFF) return HGEMM_ERR_INVALID_ARG;
  args.num_tiles = static_cast<int>(tiles);
  args.full_tiles = args.num_tiles;
  args.group_m = group_m_setting();
  args.grid = static_cast<int>(tiles < dev.num_sms ? tiles : dev.num_sms);
  args.status = t_ctx.status;
  args.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  args.inject = g_inject.load(std::memory_order_relaxed);
  args.epi = epi;
  args.C = static_cast<const uint16_t*>(g.c_src ? g.c_src : C);  // C_old, for a fused epilogue
  args.ldc = g.c_src ? g.ld_src : g.ldc;
  cudaError_t e = bn == hg::kNarrowBN ? hg::launch_tc_128x64(ma, mb, mc, args, stream)
                                      : hg::launch_tc_128x256(ma, mb, mc, args, stream);
  return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
}

// A batch of equal products in one launch of the pair kernel: product j
// (j < count) is n_each columns of C by k_each of K, with A's K, B's N and
// K, and C's N coordinates shifted by j·shift from those of the first; the
// Gemm passed with it spans them all. n_each is a multiple of the tile
// width and k_each of the K block, so no tile reaches past its product.
struct PairBatch {
  int count;
  int64_t shift, n_each, k_each;
};

// whole_tiles: never cut the last wave's tiles into column parts (a product
// computed in place needs every tile to read all the columns it writes).
int run_tc_pair(const Gemm& g, const hg::EpiArgs& epi, const DeviceState& dev,
            cudaStream_t stream, const PairBatch* batch = nullptr, bool whole_tiles = false) {
  const void* A = g.A;
  const void* B = g.B;
  void* C = g.C;
  const int64_t M = g.M, N = g.N, K = g.K;
  const int64_t n_one = batch ? batch->n_each : N, k_one = batch ? batch->k_each : K;
  hg::TcArgs args{};
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.K = static_cast<int>(K);
  args.num_m = static_cast<int>((M + 2 * hg::kTcBM - 1) / (2 * hg::kTcBM));
  args.num_n = static_cast<int>((n_one + hg::kPairBN - 1) / hg::kPairBN);
  args.num_kb = static_cast<int>((k_one + hg::kTcBK - 1) / hg::kTcBK);
  const int64_t per = static_cast<int64_t>(args.num_m) * args.num_n;
  const int64_t tiles = per * (batch ? batch->count : 1);
  if (batch) {
    args.batch_tiles = static_cast<int>(per);
    args.batch_shift = static_cast<int>(batch->shift);
  }
  if (tiles > 0x1FFFFFFF) return HGEMM_ERR_INVALID_ARG;
  const int64_t clusters = hg::pair_max_clusters(dev.num_sms);
  // Last (or only) wave: if its tiles leave at least half of the clusters
  // idle, cut them into 128-column parts, or 64-column ones when even those
  // leave half idle and the tiles' columns reach past 128 of them.
  const int64_t full_waves = tiles / clusters;
  const int64_t rest = tiles - full_waves * clusters;
  int parts = 1;
  if (!whole_tiles && tail_split_setting() && rest > 0 && 2 * rest <= clusters) {
    parts = 2;
    const int64_t last_cols = n_one - static_cast<int64_t>(args.num_n - 1) * hg::kPairBN;
    // (an N-contiguous B arrives in 64-column boxes: a CTA's share of a part
    // must be at least one box, so its parts keep 128 columns)
    if (4 * rest <= clusters && (args.num_n > 1 || last_cols > 128) && !g.b_mn) parts = 4;
  }
  args.part_cols = hg::kPairBN / parts;
  args.full_tiles = static_cast<int>(parts > 1 ? tiles - rest : tiles);
  // stages hold whole-tile operands, or a part's when every unit is a part
  args.stage_bytes = hg::kTcBM * hg::kTcBK * 2 +
                     (args.full_tiles > 0 ? hg::kPairBN / 2 : args.part_cols / 2) * hg::kTcBK * 2;
  args.stages = hg::kPairRingBytes / args.stage_bytes;
  args.num_tiles = static_cast<int>(parts > 1 ? tiles - rest + parts * rest : tiles);
  args.group_m = group_m_setting();
  args.grid = static_cast<int>(2 * (args.num_tiles < clusters ? args.num_tiles : clusters));
  args.status = t_ctx.status;
  args.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  args.inject = g_inject.load(std::memory_order_relaxed);
  args.epi = epi;
  args.C = static_cast<const uint16_t*>(g.c_src ? g.c_src : C);  // C_old, for a fused epilogue
  args.ldc = g.c_src ? g.ld_src : g.ldc;
  args.a_mn = g.a_mn ? 1 : 0;
  args.b_mn = g.b_mn ? 1 : 0;
  CUtensorMap ma, mb, mbp, mc;
  int rc;
  // MN-major operands: boxes of 64 M or N elements × 64 K rows
  if (g.a_mn)
    rc = encode_map(&ma, A, K, M, g.lda, hg::kTcBK, 64);
  else
    rc = encode_map(&ma, A, M, K, g.lda, hg::kTcBM, hg::kTcBK);
  if (rc != HGEMM_OK) return rc;
  if (g.b_mn) {
    if ((rc = encode_map(&mb, B, K, N, g.ldb, hg::kTcBK, 64)) != HGEMM_OK) return rc;
    mbp = mb;
  } else {
    if ((rc = encode_map(&mb, B, N, K, g.ldb, hg::kPairBN / 2, hg::kTcBK)) != HGEMM_OK) return rc;
    if ((rc = encode_map(&mbp, B, N, K, g.ldb, args.part_cols / 2, hg::kTcBK)) != HGEMM_OK) return rc;
  }
  if ((rc = encode_map(&mc, C, M, N, g.ldc, hg::kEpiRows, hg::kEpiCols)) != HGEMM_OK) return rc;
  cudaError_t e = hg::launch_tc_pair(ma, mb, mbp, mc, args, stream);
  return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
}

int run_tc_wide(const Gemm& g, const hg::EpiArgs& epi, const DeviceState& dev,
            cudaStream_t stream) {
  const void* A = g.A;
  const void* B = g.B;
  void* C = g.C;
  const int64_t M = g.M, N = g.N, K = g.K;
  CUtensorMap ma, mb, mc;
  int rc;
  // MN-major operands: boxes of 64 M or N elements × 64 K rows
  if ((rc = g.a_mn ? encode_map(&ma, A, K, M, g.lda, hg::kTcBK, 64)
                   : encode_map(&ma, A, M, K, g.lda, hg::kTcBM, hg::kTcBK)) != HGEMM_OK)
    return rc;
  if ((rc = g.b_mn ? encode_map(&mb, B, K, N, g.ldb, hg::kTcBK, 64)
                   : encode_map(&mb, B, N, K, g.ldb, hg::kPairBN / 2, hg::kTcBK)) != HGEMM_OK)
    return rc;
  if ((rc = encode_map(&mc, C, M, N, g.ldc, hg::kEpiRows, hg::kEpiCols)) != HGEMM_OK) return rc;
  hg::TcArgs args{};
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.K = static_cast<int>(K);
  args.num_m = static_cast<int>((M + 2 * hg::kTcBM - 1) / (2 * hg::kTcBM));
  args.num_n = static_cast<int>((N + 2 * hg::kPairBN - 1) / (2 * hg::kPairBN));
  args.num_kb = static_cast<int>((K + hg::kTcBK - 1) / hg::kTcBK);
  const int64_t tiles = static_cast<int64_t>(args.num_m) * args.num_n;
  if (tiles > 0x3FFFFFFF) return HGEMM_ERR_INVALID_ARG;
  args.num_tiles = static_cast<int>(tiles);
  args.full_tiles = args.num_tiles;
  args.group_m = group_m_setting();
  const int64_t clusters = hg::wide_max_clusters(dev.num_sms);
  args.grid = static_cast<int>(2 * (tiles < clusters ? tiles : clusters));
  args.status = t_ctx.status;
  args.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  args.inject = g_inject.load(std::memory_order_relaxed);
  args.epi = epi;
  args.C = static_cast<const uint16_t*>(g.c_src ? g.c_src : C);  // C_old, for a fused epilogue
  args.ldc = g.c_src ? g.ld_src : g.ldc;
  args.a_mn = g.a_mn ? 1 : 0;
  args.b_mn = g.b_mn ? 1 : 0;
  cudaError_t e = hg::launch_tc_wide(ma, mb, mc, args, stream);
  return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
}

int run_skinny(const Gemm& g, int split, int tile_n, const hg::EpiArgs& epi, const DeviceState& dev,
               cudaStream_t stream) {
  const void* A = g.A;
  const void* B = g.B;
  void* C = g.C;
  const int64_t M = g.M, N = g.N, K = g.K;
  CUtensorMap ma, mb, mc;
  int rc;
  // MN-major operands: boxes of 64 M or N elements × 64 K rows
  if ((rc = g.a_mn ? encode_map(&ma, A, K, M, g.lda, hg::kTcBK, 64)
                   : encode_map(&ma, A, M, K, g.lda, hg::kTcBM, hg::kTcBK)) != HGEMM_OK)
    return rc;
  if ((rc = g.b_mn ? encode_map(&mb, B, K, N, g.ldb, hg::kTcBK, 64)
                   : encode_map(&mb, B, N, K, g.ldb, tile_n / 2, hg::kTcBK)) != HGEMM_OK)
    return rc;
  if ((rc = encode_map(&mc, C, M, N, g.ldc, hg::kEpiRows, hg::kEpiCols)) != HGEMM_OK) return rc;
  hg::TcArgs args{};
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.K = static_cast<int>(K);
  args.num_m = static_cast<int>((M + 2 * hg::kTcBM - 1) / (2 * hg::kTcBM));
  args.num_n = static_cast<int>((N + tile_n - 1) / tile_n);
  args.num_kb = static_cast<int>((K + hg::kTcBK - 1) / hg::kTcBK);
  const int64_t tiles = static_cast<int64_t>(args.num_m) * args.num_n;
  if (tiles * 2 * split > 0x7FFFFFFF) return HGEMM_ERR_INVALID_ARG;
  args.num_tiles = static_cast<int>(tiles);
  args.full_tiles = args.num_tiles;
  args.group_m = 1;
  args.grid = static_cast<int>(tiles * 2 * split);
  args.status = t_ctx.status;
  args.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  args.inject = g_inject.load(std::memory_order_relaxed);
  args.epi = epi;
  args.C = static_cast<const uint16_t*>(g.c_src ? g.c_src : C);  // C_old, for a fused epilogue
  args.ldc = g.c_src ? g.ld_src : g.ldc;
  args.a_mn = g.a_mn ? 1 : 0;
  args.b_mn = g.b_mn ? 1 : 0;
  cudaError_t e = hg::launch_skinny(split, tile_n, ma, mb, mc, args, stream);
  return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
}

int dispatch(const Gemm& g, const hg::EpiArgs& epi, const DeviceState& dev, cudaStream_t stream) {
  cudaError_t e;
  int split = 1, tile_n = hg::kPairBN;
  switch (choose_path(g, dev.prof, epi.mode != 0, &split, &tile_n)) {
    case HGEMM_PATH_NONE:
      return HGEMM_OK;
    case HGEMM_PATH_ZERO:
      if (g.c_src) return HGEMM_ERR_INVALID_ARG;  // the empty sum reads C_old from C
      e = hg::launch_empty_sum(static_cast<uint16_t*>(g.C), g.M, g.N, g.ldc, epi, stream);
      return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
    case HGEMM_PATH_TC:
      return run_tc(g, epi, dev, stream, hg::kTcBN);
    case HGEMM_PATH_TC_NARROW:
      return run_tc(g, epi, dev, stream, hg::kNarrowBN);
    case HGEMM_PATH_TC_PAIR:
      return run_tc_pair(g, epi, dev, stream);
    case HGEMM_PATH_TC_WIDE:
      return run_tc_wide(g, epi, dev, stream);
    case HGEMM_PATH_SKINNY:
      return run_skinny(g, split, tile_n, epi, dev, stream);
    default: {
      if (g.c_src) return HGEMM_ERR_INVALID_ARG;  // the generic kernel reads C_old from C
      hg::PlainArgs pa{static_cast<const uint16_t*>(g.A), static_cast<const uint16_t*>(g.B),
                       static_cast<uint16_t*>(g.C), g.M, g.N, g.K, g.lda, g.ldb, g.ldc,
                       t_ctx.status, g_timeout_ns.load(), epi, g.a_mn ? 1 : 0, g.b_mn ? 1 : 0};
      e = hg::launch_generic(pa, dev.num_sms, stream);
      return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
    }
  }
}

// Helper streams and events of the host-buffer entry point, created once per
// device and kept for the life of the process (no device memory).
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  static constexpr int kEvents = 2 + 2 * 16;
  cudaEvent_t ev[kEvents] = {};
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mu;

int pipe_for_current_device(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return HGEMM_ERR_UNSUPPORTED_DEVICE;
  HostPipe& hp = g_pipes[dev];
  if (!hp.ready) {
    if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess)
      return cuda_fail(e);
    for (auto& ev : hp.ev)
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
    hp.ready = true;
  }
  *out = &hp;
  return HGEMM_OK;
}

// Helper streams of hgemm_trmm: the independent updates of one level of the
// recursion run on them concurrently (fork and join through events on the
// caller's stream). Created once per device, kept for the life of the process.
struct TrmmPipe {
  bool ready = false;
  static constexpr int kStreams = 4;
  cudaStream_t s[kStreams] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kStreams] = {};
  std::mutex mu;
};
TrmmPipe g_trmm_pipes[kMaxDevices];

int trmm_pipe(int dev, TrmmPipe** out) {
  TrmmPipe& tp = g_trmm_pipes[dev];
  if (!tp.ready) {
    cudaError_t e;
    for (auto& st : tp.s)
      if ((e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaEventCreateWithFlags(&tp.fork, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
    for (auto& ev : tp.join)
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
    tp.ready = true;
  }
  *out = &tp;
  return HGEMM_OK;
}

}  // namespace

extern "C" {

int hgemm(const hgemm_half_t* A, const hgemm_half_t* B, hgemm_half_t* C, int64_t M, int64_t N,
          int64_t K, cudaStream_t stream) {
  const Gemm g = dense(A, B, C, M, N, K);
  int rc = validate(g);
  if (rc != HGEMM_OK) return rc;
  if (M == 0 || N == 0) return HGEMM_OK;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != HGEMM_OK) return rc;
  return dispatch(g, kPlainEpilogue, *dev, stream);
}

// The fused product on a validated problem: bias checks, epilogue mode.
int run_fused(const Gemm& g, float alpha, float beta, const hgemm_half_t* bias, int relu,
              cudaStream_t stream) {
  if (bias) {
    if (reinterpret_cast<uintptr_t>(bias) & 1u) return HGEMM_ERR_INVALID_ARG;
    // C is written while bias is read
    if (g.M > 0 && g.N > 0 &&
        ranges_overlap(g.C, 2 * static_cast<uint64_t>((g.M - 1) * g.ldc + g.N), bias,
                       2 * static_cast<uint64_t>(g.N)))
      return HGEMM_ERR_ALIAS;
  }
  if (g.M == 0 || g.N == 0) return HGEMM_OK;
  hg::EpiArgs epi{alpha, beta, reinterpret_cast<const uint16_t*>(bias), relu ? 1 : 0, 0};
  epi.mode = beta != 0.0f ? 2 : ((alpha != 1.0f || bias || relu) ? 1 : 0);
  DeviceState* dev = nullptr;
  int rc;
  if ((rc = current_device(&dev)) != HGEMM_OK) return rc;
  return dispatch(g, epi, *dev, stream);
}

int hgemm_ex(const hgemm_half_t* A, const hgemm_half_t* B, hgemm_half_t* C, int64_t M, int64_t N,
             int64_t K, float alpha, float beta, const hgemm_half_t* bias, int relu,
             cudaStream_t stream) {
  const Gemm g = dense(A, B, C, M, N, K);
  const int rc = validate(g);
  if (rc != HGEMM_OK) return rc;
  return run_fused(g, alpha, beta, bias, relu, stream);
}

int hgemm_strided(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
                  hgemm_half_t* C, int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha,
                  float beta, const hgemm_half_t* bias, int relu, cudaStream_t stream) {
  const Gemm g{A, B, C, M, N, K, lda, ldb, ldc};
  const int rc = validate(g);
  if (rc != HGEMM_OK) return rc;
  return run_fused(g, alpha, beta, bias, relu, stream);
}

int hgemm_layout(int a_layout, int b_layout, const hgemm_half_t* A, int64_t lda,
                 const hgemm_half_t* B, int64_t ldb, hgemm_half_t* C, int64_t ldc, int64_t M,
                 int64_t N, int64_t K, float alpha, float beta, const hgemm_half_t* bias, int relu,
                 cudaStream_t stream) {
  if ((a_layout != HGEMM_A_ROW_MAJOR && a_layout != HGEMM_A_COL_MAJOR) ||
      (b_layout != HGEMM_B_COL_MAJOR && b_layout != HGEMM_B_ROW_MAJOR))
    return HGEMM_ERR_INVALID_ARG;
  Gemm g{A, B, C, M, N, K, lda, ldb, ldc};
  g.a_mn = a_layout == HGEMM_A_COL_MAJOR;
  g.b_mn = b_layout == HGEMM_B_ROW_MAJOR;
  const int rc = validate(g);
  if (rc != HGEMM_OK) return rc;
  return run_fused(g, alpha, beta, bias, relu, stream);
}

int hgemm_trmm(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
               hgemm_half_t* C, int64_t ldc, int64_t n, int64_t m, float alpha,
               cudaStream_t stream) {
  if (n < 0 || m < 0 || n > HGEMM_TRMM_MAX_N || m > HGEMM_MAX_DIM) return HGEMM_ERR_INVALID_ARG;
  if (n == 0 || m == 0) return HGEMM_OK;
  const int64_t ld_lim = int64_t(1) << 40;
  if (lda < n || ldb < n || ldc < n || lda > ld_lim || ldb > ld_lim || ldc > ld_lim)
    return HGEMM_ERR_INVALID_ARG;
  if (!A || !B || !C) return HGEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 1u)
    return HGEMM_ERR_INVALID_ARG;
  // column-major spans (in elements): A n×n, B and C n×m
  const unsigned __int128 sa = static_cast<unsigned __int128>(n - 1) * lda + n;
  const unsigned __int128 sb = static_cast<unsigned __int128>(m - 1) * ldb + n;
  const unsigned __int128 sc = static_cast<unsigned __int128>(m - 1) * ldc + n;
  const unsigned __int128 lim = static_cast<unsigned __int128>(1) << 61;
  if (sa >= lim || sb >= lim || sc >= lim) return HGEMM_ERR_INVALID_ARG;
  if (ranges_overlap(C, 2 * static_cast<uint64_t>(sc), A, 2 * static_cast<uint64_t>(sa)) ||
      ranges_overlap(C, 2 * static_cast<uint64_t>(sc), B, 2 * static_cast<uint64_t>(sb)))
    return HGEMM_ERR_ALIAS;
  DeviceState* dev = nullptr;
  int rc;
  if ((rc = current_device(&dev)) != HGEMM_OK) return rc;

  // The page's recursion on blocks [off, off + s) of the triangle: the
  // diagonal blocks of at most kTrmmLeaf are leaves; every larger block
  // splits at s1 (half of s rounded up to a multiple of 64, so every block
  // starts on a multiple of 64) and adds the off-diagonal update
  //   C[off : off+s1, :] += alpha · A[off+s1 : off+s, off : off+s1]ᵀ · B[off+s1 : off+s, :]
  // after both halves (post-order: the update of a block sees its first
  // half complete).
  struct Update {
    int64_t off, s1, s2;
  };
  hg::TriLeaves leaves{};
  std::vector<std::vector<Update>> levels;  // updates by depth in the recursion
  struct Frame {
    int64_t off, s;
    int depth;
  };
  std::vector<Frame> stack{{0, n, 0}};
  while (!stack.empty()) {
    const Frame f = stack.back();
    stack.pop_back();
    if (f.s <= kTrmmLeaf) {
      if (leaves.count == hg::kMaxLeaves) return HGEMM_ERR_INVALID_ARG;
      leaves.off[leaves.count] = f.off;
      leaves.size[leaves.count] = f.s;
      ++leaves.count;
      continue;
    }
    const int64_t s1 = ((f.s / 2 + 63) / 64) * 64;
    if (static_cast<int>(levels.size()) <= f.depth) levels.resize(f.depth + 1);
    levels[f.depth].push_back({f.off, s1, f.s - s1});
    stack.push_back({f.off + s1, f.s - s1, f.depth + 1});
    stack.push_back({f.off, s1, f.depth + 1});
  }

  // In the GEMM view, Cᵀ (m × n, pitch ldc) = Bᵀ (m × n, pitch ldb) · lower(A),
  // where row i of the second operand is column i of A (pitch lda).
  const hg::EpiArgs scale{alpha, 0.0f, nullptr, 0, alpha != 1.0f ? 1 : 0};
  const int forced = g_forced_path.load(std::memory_order_relaxed);
  // The leaves run on the tensor cores when every leaf order is a multiple of
  // 64 (n is) and TMA can describe the operands; otherwise (or with the
  // generic path forced) on the generic kernel, which masks as it loads.
  cudaError_t e = cudaSuccess;
  bool tc_leaves = forced != HGEMM_PATH_GENERIC && n % 64 == 0 && m <= (int64_t(1) << 30) &&
                   ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                     reinterpret_cast<uintptr_t>(C)) & 15u) == 0 &&
                   lda % 8 == 0 && ldb % 8 == 0 && ldc % 8 == 0;
  if (tc_leaves) {
    // Bᵀ (m × n, pitch ldb), the triangle's rows (column i of A, pitch lda), Cᵀ
    CUtensorMap mx, ml, mc;
    tc_leaves = encode_map(&mx, B, m, n, ldb, hg::kTcBM, hg::kTcBK) == HGEMM_OK &&
                encode_map(&ml, A, n, n, lda, 64, hg::kTcBK) == HGEMM_OK &&
                encode_map(&mc, C, m, n, ldc, hg::kEpiRows, hg::kEpiCols) == HGEMM_OK;
    if (tc_leaves) {
      hg::TcArgs args{};
      args.M = static_cast<int>(m);
      args.N = static_cast<int>(n);
      args.K = static_cast<int>(n);
      args.num_m = static_cast<int>((m + hg::kTcBM - 1) / hg::kTcBM);
      args.num_tiles = leaves.count * args.num_m;
      args.full_tiles = args.num_tiles;
      args.grid = args.num_tiles < dev->num_sms ? args.num_tiles : dev->num_sms;
      args.status = t_ctx.status;
      args.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
      args.inject = g_inject.load(std::memory_order_relaxed);
      args.epi = scale;
      args.C = reinterpret_cast<const uint16_t*>(C);
      args.ldc = ldc;
      // The update of a block adds into the leaves of its first half before
      // any larger block's update does; when it is small (kTrmmFoldMacs),
      // those leaves carry it: each leaf's product runs on over the update's K
      // columns [off+s1, off+s). Taken deepest first, the carried ranges of
      // a leaf join into one range right after it (each block's second half
      // starts where the first half around the leaf ends); if they do not
      // (checked), nothing is carried. The leaves are then launched longest
      // first.
      hg::TriLeafExt ext{};
      {
        std::vector<int64_t> end(leaves.count);
        for (int b = 0; b < leaves.count; ++b) end[b] = leaves.off[b] + leaves.size[b];
        std::vector<std::vector<Update>> kept(levels.size());
        bool joined = true;
        for (int d = static_cast<int>(levels.size()) - 1; d >= 0; --d)
          for (const Update& u : levels[d]) {
            if (m * u.s1 * u.s2 > kTrmmFoldMacs || forced >= 0) {  // a forced path takes every update
              kept[d].push_back(u);
              continue;
            }
            for (int b = 0; b < leaves.count; ++b)
              if (leaves.off[b] >= u.off && leaves.off[b] < u.off + u.s1) {
                joined = joined && end[b] == u.off + u.s1;
                end[b] = u.off + u.s1 + u.s2;
              }
          }
        if (joined) {
          levels.swap(kept);
          std::vector<int> order(leaves.count);
          for (int b = 0; b < leaves.count; ++b) order[b] = b;
          std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
            return end[x] - leaves.off[x] > end[y] - leaves.off[y];
          });
          const hg::TriLeaves by_work = leaves;
          for (int k = 0; k < leaves.count; ++k) {
            const int b = order[k];
            leaves.off[k] = by_work.off[b];
            leaves.size[k] = by_work.size[b];
            ext.ext[k] = static_cast<int32_t>(end[b] - by_work.off[b] - by_work.size[b]);
          }
        }
      }
      e = hg::launch_tri_leaves_tc(mx, ml, mc, args, leaves, ext, stream);
    }
  }
  if (!tc_leaves) {
    hg::PlainArgs pa{reinterpret_cast<const uint16_t*>(B), reinterpret_cast<const uint16_t*>(A),
                     reinterpret_cast<uint16_t*>(C), m, n, n, ldb, lda, ldc,
                     t_ctx.status, g_timeout_ns.load(), scale};
    e = hg::launch_tri_leaves(pa, leaves, dev->num_sms, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);

  // Updates, deepest level first: an update reads the first half of its
  // block complete, which every deeper level and the leaves have made. The
  // updates of one level touch disjoint rows of C and run concurrently.
  const hg::EpiArgs accumulate{alpha, 1.0f, nullptr, 0, 2};
  auto issue = [&](const Update& u, cudaStream_t st) {
    const Gemm g{B + u.off + u.s1, A + u.off * lda + u.off + u.s1, C + u.off, m, u.s1, u.s2,
                 ldb, lda, ldc};
    const int r = validate(g);
    return r != HGEMM_OK ? r : dispatch(g, accumulate, *dev, st);
  };
  // A level of equal updates at a constant stride (every level when n is a
  // power of two times 256), whose updates are whole 256-column tiles and
  // whole K blocks, runs as one batched launch of the pair kernel on the
  // caller's stream; other levels run update by update on helper streams.
  auto batch_of = [&](const std::vector<Update>& lv, Gemm* span, PairBatch* pb) {
    if (lv.size() < 2 || (forced >= 0 && forced != HGEMM_PATH_TC_PAIR)) return false;
    const Update& u0 = lv[0];
    const int64_t shift = lv[1].off - u0.off;
    if (u0.s1 % hg::kPairBN != 0 || u0.s2 % hg::kTcBK != 0 || shift <= 0) return false;
    for (size_t k = 1; k < lv.size(); ++k)
      if (lv[k].s1 != u0.s1 || lv[k].s2 != u0.s2 || lv[k].off != u0.off + static_cast<int64_t>(k) * shift)
        return false;
    const int64_t cnt = static_cast<int64_t>(lv.size());
    *span = Gemm{B + u0.off + u0.s1, A + u0.off * lda + u0.off + u0.s1, C + u0.off, m,
                 (cnt - 1) * shift + u0.s1, (cnt - 1) * shift + u0.s2, ldb, lda, ldc};
    *pb = PairBatch{static_cast<int>(cnt), shift, u0.s1, u0.s2};
    return tma_ok(*span) && validate(*span) == HGEMM_OK;
  };
  TrmmPipe* tp = nullptr;
  bool need_pipe = false;
  for (const auto& lv : levels) {
    Gemm span{};
    PairBatch pb{};
    need_pipe = need_pipe || (lv.size() > 1 && !batch_of(lv, &span, &pb));
  }
  if (need_pipe && (rc = trmm_pipe(dev->id, &tp)) != HGEMM_OK) return rc;
  std::unique_lock<std::mutex> lock;
  if (tp) lock = std::unique_lock<std::mutex>(tp->mu);
  for (int d = static_cast<int>(levels.size()) - 1; d >= 0; --d) {
    const auto& lv = levels[d];
    if (lv.empty()) continue;  // every update of the level carried by a leaf
    if (lv.size() == 1) {
      if ((rc = issue(lv[0], stream)) != HGEMM_OK) return rc;
      continue;
    }
    Gemm span{};
    PairBatch pb{};
    if (batch_of(lv, &span, &pb)) {
      if ((rc = run_tc_pair(span, accumulate, *dev, stream, &pb)) != HGEMM_OK) return rc;
      continue;
    }
    const int used = static_cast<int>(lv.size() < TrmmPipe::kStreams ? lv.size() : TrmmPipe::kStreams);
    if ((e = cudaEventRecord(tp->fork, stream)) != cudaSuccess) return cuda_fail(e);
    for (int i = 0; i < used; ++i)
      if ((e = cudaStreamWaitEvent(tp->s[i], tp->fork, 0)) != cudaSuccess) return cuda_fail(e);
    for (size_t k = 0; k < lv.size(); ++k)
      if ((rc = issue(lv[k], tp->s[k % used])) != HGEMM_OK) return rc;
    for (int i = 0; i < used; ++i) {
      if ((e = cudaEventRecord(tp->join[i], tp->s[i])) != cudaSuccess) return cuda_fail(e);
      if ((e = cudaStreamWaitEvent(stream, tp->join[i], 0)) != cudaSuccess) return cuda_fail(e);
    }
  }
  return HGEMM_OK;
}

namespace {

// The diagonal blocks of order ≤ leaf of the TRSM recursion in the order it
// solves them (second half first; first half first when fwd); false when
// there are more than the table holds.
bool trsm_leaves(int64_t n, int64_t leaf, hg::TriLeaves* leaves, bool fwd = false) {
  leaves->count = 0;
  std::function<bool(int64_t, int64_t)> walk = [&](int64_t off, int64_t s) -> bool {
    if (s <= leaf) {
      if (leaves->count == hg::kMaxLeaves) return false;
      leaves->off[leaves->count] = off;
      leaves->size[leaves->count] = s;
      ++leaves->count;
      return true;
    }
    const int64_t s1 = ((s / 2 + 63) / 64) * 64;
    return fwd ? (walk(off, s1) && walk(off + s1, s - s1)) : (walk(off + s1, s - s1) && walk(off, s1));
  };
  return n > 0 && walk(0, n);
}

// Largest number of right-hand sides for which hgemm_trsm_ws takes the chain
// schedule by itself.
constexpr int64_t kChainAutoMaxM = 1024;

// one inverse in the workspace: FP16, kTrsmInverseLeaf² (512 KiB)
constexpr uint64_t kTrsmInverseBytes = 2ull * hg::kTrsmInverseLeaf * hg::kTrsmInverseLeaf;

// ---- the chain schedule's plan (see hgemm_trsm_chain.cu)
//
// Cost model of a tile (measured on the chain kernel): an MMA issuer takes
// ~0.24 µs per 64-deep K step of an N ≤ 128 tile (~61-65 cycles per
// M=128 MMA instruction whatever N up to 128, plus its wait) and ~0.40 µs at
// N = 256; an SM takes in operands at ~100 GB/s, (bm + bn)·128 bytes per
// step. A phase costs the longest CTA's tiles plus ~3 µs of barrier, launch
// of the first copies and epilogue.
double chain_step_us(int bm, int bn) {
  const double mma = bn <= 128 ? 0.24 : 0.40;
  const double intake = (bm + bn) * 128.0 / 1.0e5;
  return mma > intake ? mma : intake;
}
constexpr double kChainPhaseUs = 3.0;

struct ChainTile {
  int bm, bn, tiles;
  double us;  // one tile
};

// The tile shapes of a group of rows × ncols outputs with ksteps K steps.
int chain_tiles(int64_t rows, int64_t ncols, int ksteps, ChainTile (&out)[6]) {
  static constexpr int kBm[2] = {128, 64};
  static constexpr int kBn[3] = {256, 128, 64};
  int n = 0;
  for (int i : kBm)
    for (int j : kBn)
      out[n++] = ChainTile{i, j, static_cast<int>(((rows + i - 1) / i) * ((ncols + j - 1) / j)),
                           ksteps * chain_step_us(i, j)};
  return n;
}

// Best shapes for a phase's non-critical groups (couplings, updates: either
// may be absent, rows 0) on `span` CTAs: the longest CTA's time.
double chain_others(int64_t c_rows, int64_t c_cols, int c_steps, int64_t u_rows, int64_t u_cols, int u_steps,
                    int span, ChainTile* c_best, ChainTile* u_best) {
  ChainTile ct[6], ut[6];
  const int nc = c_rows > 0 ? chain_tiles(c_rows, c_cols, c_steps, ct) : 1;
  const int nu = u_rows > 0 ? chain_tiles(u_rows, u_cols, u_steps, ut) : 1;
  if (c_rows <= 0) ct[0] = ChainTile{0, 0, 0, 0.0};
  if (u_rows <= 0) ut[0] = ChainTile{0, 0, 0, 0.0};
  double best = -1.0;
  for (int a = 0; a < nc; ++a) {
    if (c_rows > 0 && ct[a].bm != 128) continue;  // a coupling's rows are a whole block: 128-row tiles
    for (int b = 0; b < nu; ++b) {
      const int tiles = ct[a].tiles + ut[b].tiles;
      const int waves = span > 0 ? (tiles + span - 1) / span : (tiles > 0 ? 1 << 20 : 0);
      const double t = waves * (ct[a].us > ut[b].us ? ct[a].us : ut[b].us);
      if (best < 0 || t < best - 1e-9) {
        best = t;
        *c_best = ct[a];
        *u_best = ut[b];
      }
    }
  }
  return best;
}

// Plans the chain launch of a solve whose inverses are (or will be) in
// slots 0 .. count-1 of W, with slot `count` spare, as one of two plans:
//  fused (one phase per block, k in the order of the solve):
//   products of block k (critical: CTAs of their own), K segments for
//     L_k⁻¹ (· L_k⁻ᵀ for A·X = B) and, from the second block on, M_k;
//   couplings M_{k+1} = −C(k, k+1)·L_{k+1}⁻¹ into slot k-1 (M_1: the spare
//     slot), a slot whose inverse the solve has used;
//   updates of every block after k from Xᵀ_{k−1} (from the second block on);
//  split (two phases per block): the products of block k by L_k⁻¹ alone,
//   then the update of every block after it from Xᵀ_k.
// The plan with the lower modelled time is taken (plan: 0 either, 1 fused,
// 2 split). scale: X must become alpha·B first (not in place, or alpha !=
// 1); fold: B suits TMA and alpha != 0, so the first phases read B
// themselves instead of a copy phase: the first block's product reads B
// (scale alpha); fused, the second block's product reads B_1 and M_1 / alpha
// (scale alpha); the first update subtracts from alpha·B. Returns 0 when the
// chain does not apply (too many blocks or rows, products wider than the
// grid), else the plan taken.
int chain_plan(const hg::TriLeaves& leaves, int64_t n, int64_t m, bool scale, bool fold, float alpha, bool fwd,
               int max_grid, int plan, hg::ChainArgs* args, int* grid, int* ragged) {
  const int nb = leaves.count;
  if (nb < 1 || nb > hg::kChainMaxLeaves || max_grid < 2) return 0;
  if (m < 1 || (m + 63) / 64 > hg::kChainMaxRowGroups || n > (int64_t(1) << 30)) return 0;
  const int64_t L = hg::kTrsmInverseLeaf;
  fold = fold && scale;
  *ragged = -1;
  for (int b = 0; b < nb; ++b)
    if (leaves.size[b] % 64 != 0) {
      // only the block that ends at n (the edge of every map) may be ragged
      if (leaves.off[b] + leaves.size[b] != n || *ragged >= 0) return 0;
      *ragged = b;
    }
  auto steps = [](int64_t s) { return static_cast<int>((s + 63) / 64); };
  // the columns of the blocks after k: [0, off_k) for Aᵀ·X = B, [off_k + s_k, n) for A·X = B
  auto after = [&](int k, int64_t* u0, int64_t* u1) {
    *u0 = fwd ? leaves.off[k] + leaves.size[k] : 0;
    *u1 = fwd ? n : leaves.off[k];
  };
  // The fused plan's shapes per phase, and its modelled time.
  struct FusedPhase {
    ChainTile prod, coup, upd;
  };
  FusedPhase fp[hg::kChainMaxLeaves];
  double t_fused = 0.0;
  bool fused_ok = true;
  for (int k = 0; k < nb && fused_ok; ++k) {
    const int64_t sz = leaves.size[k];
    const int kall = steps(sz) + (k >= 1 ? steps(leaves.size[k - 1]) : 0);
    ChainTile pt[6];
    const int np = chain_tiles(m, sz, kall, pt);
    int64_t u0 = 0, u1 = 0;
    if (k >= 1) after(k, &u0, &u1);
    const bool coup = k + 1 < nb, upd = k >= 1 && u1 > u0;
    double best = -1.0;
    for (int a = 0; a < np; ++a) {
      if (pt[a].tiles > max_grid - ((coup || upd) ? 1 : 0)) continue;
      ChainTile c{}, u{};
      const double others =
          (coup || upd) ? chain_others(coup ? sz : 0, coup ? leaves.size[k + 1] : 0, coup ? steps(leaves.size[k + 1]) : 0,
                                       upd ? m : 0, u1 - u0, k >= 1 ? steps(leaves.size[k - 1]) : 0,
                                       max_grid - pt[a].tiles, &c, &u)
                        : 0.0;
      const double t = pt[a].us > others ? pt[a].us : others;
      if (best < 0 || t < best - 1e-9) {
        best = t;
        fp[k] = FusedPhase{pt[a], c, u};
      }
    }
    if (best < 0) fused_ok = false;
    t_fused += best + kChainPhaseUs;
  }
  // The split plan's shapes and time.
  FusedPhase sp[hg::kChainMaxLeaves];
  double t_split = 0.0;
  bool split_ok = true;
  for (int k = 0; k < nb && split_ok; ++k) {
    const int64_t sz = leaves.size[k];
    ChainTile pt[6];
    const int np = chain_tiles(m, sz, steps(sz), pt);
    double best = -1.0;
    for (int a = 0; a < np; ++a) {
      if (pt[a].tiles > max_grid) continue;
      const double t = pt[a].us * ((pt[a].tiles + max_grid - 1) / max_grid);
      if (best < 0 || t < best - 1e-9) {
        best = t;
        sp[k].prod = pt[a];
      }
    }
    if (best < 0) split_ok = false;
    t_split += best + kChainPhaseUs;
    int64_t u0 = 0, u1 = 0;
    after(k, &u0, &u1);
    if (u1 > u0) {
      ChainTile c{}, u{};
      t_split += chain_others(0, 0, 0, m, u1 - u0, steps(sz), max_grid, &c, &u) + kChainPhaseUs;
      sp[k].upd = u;
    }
  }
  if (plan == 1 && !fused_ok) return 0;
  if (plan == 2 && !split_ok) return 0;
  if (!fused_ok && !split_ok) return 0;
  const bool fused = plan == 1 || (plan == 0 && fused_ok && (!split_ok || t_fused <= t_split));

  int ng = 0, max_tiles = 1;
  uint32_t target = 0;
  auto mslot = [&](int k) { return k == 1 ? nb : k - 2; };  // where M_k lives
  auto group_flags = [](int kind, int a_map, int a_mn, int b_map, int b_mn, const ChainTile& t, int old_from_b,
                        int critical) {
    return hg::chain_group_flags(kind, a_map, a_mn, b_map, b_mn, t.bm, t.bn, old_from_b, 0, critical);
  };
  auto end_phase = [&](int tiles) {
    args->group[ng - 1].flags |= 1u << 16;  // the phase's last group
    max_tiles = std::max(max_tiles, tiles);
  };
  if (scale && !fold) {
    args->group[ng++] = hg::ChainGroup{hg::chain_group_flags(hg::kChainCopy, 0, 0, 0, 0, 0, 0, 0, 0, 0), 0, 0, 0, 0,
                                       0, 0, 0, 0, 0, 0, 0, -1, 1.0f, 0};
    end_phase(1);
  }
  for (int k = 0; k < nb; ++k) {
    const int64_t off = leaves.off[k], sz = leaves.size[k];
    const bool rag = k == *ragged;
    const int wbase = rag ? 0 : static_cast<int>(k * L);
    const int wmap = rag ? hg::kChainMapWRagged : hg::kChainMapW;
    const FusedPhase& f = fused ? fp[k] : sp[k];
    // the products (critical)
    const int64_t pn = (sz + f.prod.bn - 1) / f.prod.bn;
    target += static_cast<uint32_t>(pn);
    const bool from_b = fold && (k == 0 || (fused && k == 1));
    hg::ChainGroup prod{group_flags(hg::kChainProduct, from_b ? hg::kChainMapB : hg::kChainMapX, 0, wmap, fwd ? 0 : 1,
                                    f.prod, 0, 1),
                        static_cast<int>(m), static_cast<int>(off), static_cast<int>(off + sz),
                        static_cast<int>(off), 0, steps(sz), fwd ? 0 : wbase, fwd ? wbase : 0, 0, 0, 0, -1,
                        from_b ? alpha : 1.0f, target};
    if (fused && k >= 1) {
      prod.a2_kbase = static_cast<int>(leaves.off[k - 1]);
      prod.b2_kbase = static_cast<int>(mslot(k) * L);
      prod.ksteps2 = steps(leaves.size[k - 1]);
    }
    args->group[ng++] = prod;
    int tiles_phase = f.prod.tiles;
    if (fused) {
      // the coupling of block k to block k+1: rows i of block k, K and N over
      // block k+1. Aᵀ·X = B: C(i, j) = A(off_k + i, off_{k+1} + j), M-contiguous;
      // A·X = B: C(i, j) = A(off_{k+1} + j, off_k + i), K-contiguous.
      if (k + 1 < nb) {
        const int64_t no = leaves.off[k + 1], ns = leaves.size[k + 1];
        const bool rag1 = k + 1 == *ragged;
        const int wb1 = rag1 ? 0 : static_cast<int>((k + 1) * L);
        args->group[ng++] = hg::ChainGroup{
            group_flags(hg::kChainCoupling, hg::kChainMapA, fwd ? 0 : 1, rag1 ? hg::kChainMapWRagged : hg::kChainMapW,
                        fwd ? 0 : 1, f.coup, 0, 0),
            static_cast<int>(sz), 0, static_cast<int>(ns), static_cast<int>(no), static_cast<int>(off), steps(ns),
            fwd ? 0 : wb1, fwd ? wb1 : 0, 0, 0, 0, mslot(k + 1), fold && k == 0 ? -1.0f / alpha : -1.0f, 0};
        tiles_phase += f.coup.tiles;
      }
    }
    // the update from block j (fused: k-1, split: k, in a phase of its own)
    // of every block after k. Aᵀ·X = B: columns [0, off_k) minus Xᵀ_j ·
    // A(block j rows, those columns), A read K-contiguous; A·X = B: columns
    // [off_k + s_k, n) minus Xᵀ_j · A(those rows, block j columns)ᵀ, A read
    // N-contiguous.
    const int jb = fused ? k - 1 : k;
    int64_t u0 = 0, u1 = 0;
    after(k, &u0, &u1);
    if (jb >= 0 && u1 > u0) {
      if (!fused) {
        end_phase(tiles_phase);
        tiles_phase = 0;
      }
      const int64_t po = leaves.off[jb], ps = leaves.size[jb];
      args->group[ng++] = hg::ChainGroup{
          group_flags(hg::kChainUpdate, hg::kChainMapX, 0, hg::kChainMapA, fwd ? 1 : 0, f.upd,
                      fold && jb == 0 ? 1 : 0, 0),
          static_cast<int>(m), static_cast<int>(u0), static_cast<int>(u1), static_cast<int>(po), 0, steps(ps),
          static_cast<int>(po), static_cast<int>(u0), 0, 0, 0, -1, 1.0f, 0};
      tiles_phase += f.upd.tiles;
    }
    end_phase(tiles_phase);
  }
  args->num_groups = ng;
  *grid = std::min(max_grid, max_tiles);
  return fused ? 1 : 2;
}

// hgemm_trsm, hgemm_trsm_ws and hgemm_trsm_op: W (may be null) holds room
// for the inverses of the diagonal blocks. fwd: the literal orientation
// A·X = alpha·B (forward); otherwise Aᵀ·X = alpha·B.
int trsm_impl(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb, hgemm_half_t* X,
              int64_t ldx, int64_t n, int64_t m, float alpha, uint16_t* W, uint64_t w_bytes, cudaStream_t stream,
              bool fwd = false) {
  if (n < 0 || m < 0 || n > HGEMM_MAX_DIM || m > HGEMM_MAX_DIM) return HGEMM_ERR_INVALID_ARG;
  if (n == 0 || m == 0) return HGEMM_OK;
  const int64_t ld_lim = int64_t(1) << 40;
  if (lda < n || ldb < n || ldx < n || lda > ld_lim || ldb > ld_lim || ldx > ld_lim)
    return HGEMM_ERR_INVALID_ARG;
  if (!A || !B || !X) return HGEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(X)) & 1u)
    return HGEMM_ERR_INVALID_ARG;
  // column-major spans (in elements): A n×n, B and X n×m
  const unsigned __int128 sa = static_cast<unsigned __int128>(n - 1) * lda + n;
  const unsigned __int128 sb = static_cast<unsigned __int128>(m - 1) * ldb + n;
  const unsigned __int128 sx = static_cast<unsigned __int128>(m - 1) * ldx + n;
  const unsigned __int128 lim = static_cast<unsigned __int128>(1) << 61;
  if (sa >= lim || sb >= lim || sx >= lim) return HGEMM_ERR_INVALID_ARG;
  const bool in_place = static_cast<const void*>(X) == static_cast<const void*>(B) && ldx == ldb;
  if (ranges_overlap(X, 2 * static_cast<uint64_t>(sx), A, 2 * static_cast<uint64_t>(sa)) ||
      (!in_place && ranges_overlap(X, 2 * static_cast<uint64_t>(sx), B, 2 * static_cast<uint64_t>(sb))))
    return HGEMM_ERR_ALIAS;
  hg::TriLeaves leaves{};
  uint64_t inv_bytes = 0;  // the inverses' part of the workspace
  uint64_t full_bytes = 0; // with the spare slot and the synchronisation words
  if (W) {
    if (!trsm_leaves(n, hg::kTrsmInverseLeaf, &leaves, fwd) ||
        w_bytes < kTrsmInverseBytes * static_cast<uint64_t>(leaves.count) ||
        (reinterpret_cast<uintptr_t>(W) & 15u))
      return HGEMM_ERR_INVALID_ARG;
    inv_bytes = kTrsmInverseBytes * static_cast<uint64_t>(leaves.count);
    full_bytes = inv_bytes + kTrsmInverseBytes + hg::kChainSyncBytes;
    const uint64_t wb = std::min<uint64_t>(w_bytes, full_bytes);
    if (ranges_overlap(W, wb, A, 2 * static_cast<uint64_t>(sa)) ||
        ranges_overlap(W, wb, B, 2 * static_cast<uint64_t>(sb)) ||
        ranges_overlap(W, wb, X, 2 * static_cast<uint64_t>(sx)))
      return HGEMM_ERR_ALIAS;
  }
  DeviceState* dev = nullptr;
  int rc;
  if ((rc = current_device(&dev)) != HGEMM_OK) return rc;

  uint16_t* x = reinterpret_cast<uint16_t*>(X);
  const uint16_t* a = reinterpret_cast<const uint16_t*>(A);
  cudaError_t e;
  bool chained = false;  // a launch of this solve is already on the stream
  // With a workspace, the recursion stops at blocks of order ≤
  // kTrsmInverseLeaf, each solved as an in-place tensor-core product by its
  // inverse (all inverses computed in one launch first): X_bᵀ := X_bᵀ · L_b⁻¹.
  // X must suit TMA. Measured at n = m = 8192: substitution for the blocks of
  // 256, 1.30 ms; products by the inverses of the blocks of 256, 0.89 ms.
  const bool by_inverse = W && (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && ldx % 8 == 0 &&
                          g_forced_path.load(std::memory_order_relaxed) < 0;
  t_trsm_schedule = by_inverse ? HGEMM_TRSM_RECURSIVE : HGEMM_TRSM_SUBSTITUTION;
  // The chain: everything after the inverses in one persistent launch (the
  // workspace's synchronisation words after the inverses, the triangle
  // suited to TMA).
  // Automatic choice: the chain for at most kChainAutoMaxM right-hand sides,
  // where its one launch beats the recursion's chain of launches (measured);
  // past that the recursion's large products are faster.
  const int schedule = g_trsm_schedule.load(std::memory_order_relaxed);
  const bool b_tma = (reinterpret_cast<uintptr_t>(B) & 15u) == 0 && ldb % 8 == 0;
  hg::ChainArgs chain{};
  int chain_grid = 0, ragged = -1;
  const bool forced_chain = schedule == HGEMM_TRSM_CHAIN || schedule == HGEMM_TRSM_CHAIN_FUSED ||
                            schedule == HGEMM_TRSM_CHAIN_SPLIT;
  const int plan = schedule == HGEMM_TRSM_CHAIN_FUSED ? 1 : schedule == HGEMM_TRSM_CHAIN_SPLIT ? 2 : 0;
  int planned = 0;
  const bool use_chain = by_inverse && schedule != HGEMM_TRSM_RECURSIVE && (forced_chain || m <= kChainAutoMaxM) &&
                         w_bytes >= full_bytes && (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 8 == 0 &&
                         (planned = chain_plan(leaves, n, m, !in_place || alpha != 1.0f, b_tma && alpha != 0.0f,
                                               alpha, fwd, hg::chain_max_grid(dev->num_sms), plan, &chain,
                                               &chain_grid, &ragged)) != 0;
  uint32_t* sync = use_chain ? reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(W) + inv_bytes +
                                                           kTrsmInverseBytes)
                             : nullptr;
  if (by_inverse) {
    e = hg::launch_trsm_inverse(a, lda, W, leaves, sync, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    chained = true;
  }
  if (use_chain) {
    CUtensorMap mx, mb, mw, mwr, ma;
    const int64_t L = hg::kTrsmInverseLeaf;
    if ((rc = encode_map(&mx, x, m, n, ldx, 64, 64)) != HGEMM_OK ||
        (rc = b_tma ? encode_map(&mb, B, m, n, ldb, 64, 64) : encode_map(&mb, x, m, n, ldx, 64, 64)) != HGEMM_OK ||
        (rc = encode_map(&mw, W, static_cast<int64_t>(leaves.count + 1) * L, L, L, 64, 64)) != HGEMM_OK ||
        (rc = encode_map(&ma, a, n, n, lda, 64, 64)) != HGEMM_OK)
      return rc;
    mwr = mw;
    if (ragged >= 0 && (rc = encode_map(&mwr, W + ragged * L * L, leaves.size[ragged], leaves.size[ragged], L,
                                        64, 64)) != HGEMM_OK)
      return rc;
    chain.X = x;
    chain.ldx = ldx;
    chain.B = reinterpret_cast<const uint16_t*>(B);
    chain.ldb = ldb;
    chain.W = W;
    chain.alpha = alpha;
    chain.m = static_cast<int>(m);
    chain.n = static_cast<int>(n);
    chain.copy_vec = n % 8 == 0 && ldb % 8 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    chain.sync = sync;
    chain.status = t_ctx.status;
    chain.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    chain.inject = g_inject.load(std::memory_order_relaxed);
    e = hg::launch_trsm_chain(mx, mb, mw, mwr, ma, chain, chain_grid, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    t_trsm_schedule = planned == 1 ? HGEMM_TRSM_CHAIN_FUSED : HGEMM_TRSM_CHAIN_SPLIT;
    return HGEMM_OK;
  }
  int leaf_index = 0;  // position in `leaves` (the order of the solve)
  // X := alpha·B, folded into the solve when it goes by the inverses and B
  // suits TMA: the first write of every row block of X is then either its
  // product by the inverse, reading alpha·B (the block the recursion reaches
  // first), or an update that reads alpha·B as C_old (its first half, or
  // second forward); a block solved by substitution copies its rows first.
  // Otherwise one scaled copy of all of B first.
  const bool b_src = (reinterpret_cast<uintptr_t>(B) & 15u) == 0 && ldb % 8 == 0;
  const bool fold = by_inverse && b_src && (!in_place || alpha != 1.0f);
  const uint16_t* bsrc = reinterpret_cast<const uint16_t*>(B);
  if (!fold && (!in_place || alpha != 1.0f)) {
    e = hg::launch_scale_copy(bsrc, ldb, x, ldx, n, m, alpha, dev->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    chained = true;
  }
  // The update of block [off, off + s) split at s1, in the GEMM view:
  //   X1ᵀ (m × s1, pitch ldx) -= X2ᵀ (m × s2, pitch ldx) · A21 (s2 × s1),
  // where column i of A21 is A[off+s1 : off+s, off+i] (pitch lda). The
  // product reads columns [off+s1, off+s) of X and writes [off, off+s1):
  // the element sets are disjoint, so the span check of validate(), which
  // sees the interleaved columns as an overlap, is not applied.
  // Forward (A·X = B): X2ᵀ (m × s2) -= X1ᵀ (m × s1) · A21ᵀ (s1 × s2), where
  // row k of A21ᵀ is A[off+s1 : off+s, off+k], contiguous (an N-contiguous
  // second operand, pitch lda); it reads [off, off+s1) and writes
  // [off+s1, off+s).
  const hg::EpiArgs subtract{-1.0f, 1.0f, nullptr, 0, 2};
  // the first write of a row block when the copy is folded: alpha·B - product
  const hg::EpiArgs subtract_from_b{-1.0f, alpha, nullptr, 0, 2};
  const hg::EpiArgs scale_b{alpha, 0.0f, nullptr, 0, alpha != 1.0f ? 1 : 0};
  // The page's recursion, second half first: every row of a block depends on
  // the rows below it (forward: first half first, on the rows above).
  // inverse: the block's inverse is in the workspace (a block of the
  // inverse-product recursion); otherwise the blocks of order ≤ kTrsmLeaf
  // are solved by substitution.
  // fresh: rows [off, off + s) of X not yet written (alpha·B not yet copied)
  std::function<int(int64_t, int64_t, bool, bool)> solve = [&](int64_t off, int64_t s, bool inverse,
                                                               bool fresh) -> int {
    if (inverse && s <= hg::kTrsmInverseLeaf) {
      const int b = leaf_index++;
      if (s % 8 == 0) {
        // Xᵀ[:, off : off+s] (m × s, pitch ldx) := itself · L⁻¹, where row k of
        // L⁻¹ is contiguous in W_b (an N-contiguous second operand, pitch
        // kTrsmInverseLeaf). A tile of 256 rows × all s ≤ 512 columns (the wide
        // kernel's, or the pair kernel's for s ≤ 256, never cut into column
        // parts) reads every column it writes and no other tile reads them,
        // so the product runs in place.
        // forward: X_bᵀ := X_bᵀ · L⁻ᵀ, whose column j is row j of L⁻¹: the
        // same workspace read as a K-contiguous second operand
        // fresh: X_bᵀ := alpha·B_bᵀ · L⁻¹, the first operand read from B
        Gemm g{fresh ? static_cast<const void*>(bsrc + off) : static_cast<const void*>(x + off),
               W + static_cast<int64_t>(b) * hg::kTrsmInverseLeaf * hg::kTrsmInverseLeaf, x + off, m,
               s, s, fresh ? ldb : ldx, hg::kTrsmInverseLeaf, ldx};
        g.b_mn = !fwd;
        chained = true;
        const hg::EpiArgs& epi = fresh ? scale_b : kPlainEpilogue;
        return s > hg::kPairBN ? run_tc_wide(g, epi, *dev, stream)
                               : run_tc_pair(g, epi, *dev, stream, nullptr, true);
      }
      // order not a multiple of 8: this block by substitution
      return solve(off, s, false, fresh);
    }
    if (s <= hg::kTrsmLeaf) {
      if (fresh) {
        // the substitution works in place: this block's rows of alpha·B first
        e = hg::launch_scale_copy(bsrc + off, ldb, x + off, ldx, s, m, alpha, dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        chained = true;
      }
      const cudaError_t le = hg::launch_trsm_leaf(a, lda, x, ldx, off, static_cast<int>(s), m,
                                                  dev->num_sms, chained, fwd, stream);
      chained = true;
      return le == cudaSuccess ? HGEMM_OK : cuda_fail(le);
    }
    const int64_t s1 = ((s / 2 + 63) / 64) * 64, s2 = s - s1;
    if (fwd) {
      int r = solve(off, s1, inverse, fresh);
      if (r != HGEMM_OK) return r;
      Gemm g{x + off, a + off * lda + off + s1, x + off + s1, m, s2, s1, ldx, lda, ldx};
      g.b_mn = true;
      if (fresh) {
        g.c_src = bsrc + off + s1;
        g.ld_src = ldb;
      }
      if ((r = dispatch(g, fresh ? subtract_from_b : subtract, *dev, stream)) != HGEMM_OK) return r;
      return solve(off + s1, s2, inverse, false);
    }
    int r = solve(off + s1, s2, inverse, fresh);
    if (r != HGEMM_OK) return r;
    Gemm g{x + off + s1, a + off * lda + off + s1, x + off, m, s1, s2, ldx, lda, ldx};
    if (fresh) {
      g.c_src = bsrc + off;
      g.ld_src = ldb;
    }
    if ((r = dispatch(g, fresh ? subtract_from_b : subtract, *dev, stream)) != HGEMM_OK) return r;
    return solve(off, s1, inverse, false);
  };
  return solve(0, n, by_inverse, fold);
}

}  // namespace

int hgemm_trsm(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
               hgemm_half_t* X, int64_t ldx, int64_t n, int64_t m, float alpha,
               cudaStream_t stream) {
  return trsm_impl(A, lda, B, ldb, X, ldx, n, m, alpha, nullptr, 0, stream);
}

size_t hgemm_trsm_workspace_size(int64_t n) {
  hg::TriLeaves leaves{};
  if (n <= 0 || n > HGEMM_MAX_DIM || !trsm_leaves(n, hg::kTrsmInverseLeaf, &leaves)) return 0;
  return static_cast<size_t>(kTrsmInverseBytes * static_cast<uint64_t>(leaves.count + 1) + hg::kChainSyncBytes);
}

int hgemm_trsm_ws(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
                  hgemm_half_t* X, int64_t ldx, int64_t n, int64_t m, float alpha, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace) return HGEMM_ERR_INVALID_ARG;
  return trsm_impl(A, lda, B, ldb, X, ldx, n, m, alpha, static_cast<uint16_t*>(workspace), workspace_bytes,
                   stream);
}

int hgemm_trsm_op(int op, const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
                  hgemm_half_t* X, int64_t ldx, int64_t n, int64_t m, float alpha, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
  if (op != HGEMM_OP_N && op != HGEMM_OP_T) return HGEMM_ERR_INVALID_ARG;
  if (!workspace && workspace_bytes != 0) return HGEMM_ERR_INVALID_ARG;
  return trsm_impl(A, lda, B, ldb, X, ldx, n, m, alpha, static_cast<uint16_t*>(workspace), workspace_bytes,
                   stream, op == HGEMM_OP_N);
}

// ---------------------------------------------------------------------------
// hgemm_trsm_noalloc: hgemm_trsm_ws for callers that cannot allocate device
// memory. Its workspace is this fixed array, part of the library's module on
// every device that loads it (8 MiB there until the process exits). In host
// code the name g_trsm_noalloc_scratch stands for a host-side shadow, not the
// device memory, so the array's device address is taken once per device with
// cudaGetSymbolAddress (with that device current) and passed on.
namespace {

__device__ __align__(256) uint16_t g_trsm_noalloc_scratch[HGEMM_TRSM_NOALLOC_MAX_BYTES / 2];

}  // namespace

int hgemm_trsm_noalloc(const hgemm_half_t* A, int64_t lda, const hgemm_half_t* B, int64_t ldb,
                       hgemm_half_t* X, int64_t ldx, int64_t n, int64_t m, float alpha, cudaStream_t stream) {
  if (n < 0 || m < 0) return HGEMM_ERR_INVALID_ARG;
  if (n == 0 || m == 0) return HGEMM_OK;
  const size_t need = hgemm_trsm_workspace_size(n);
  if (need == 0 || need > HGEMM_TRSM_NOALLOC_MAX_BYTES) return HGEMM_ERR_INVALID_ARG;
  // the device check (sm_103) first; it also binds the device's context to
  // this thread and refreshes t_ctx when that context changed
  DeviceState* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc != HGEMM_OK) return rc;
  if (!t_ctx.noalloc) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_trsm_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    t_ctx.noalloc = p;
  }
  return hgemm_trsm_ws(A, lda, B, ldb, X, ldx, n, m, alpha, t_ctx.noalloc, HGEMM_TRSM_NOALLOC_MAX_BYTES,
                       stream);
}

int hgemm_host(const hgemm_half_t* hA, const hgemm_half_t* hB, hgemm_half_t* hC, int64_t M,
               int64_t N, int64_t K, hgemm_half_t* dA, hgemm_half_t* dB, hgemm_half_t* dC,
               cudaStream_t stream) {
  int rc = validate(dense(dA, dB, dC, M, N, K));
  if (rc != HGEMM_OK) return rc;
  if ((M * K && !hA) || (N * K && !hB) || (M * N && !hC)) return HGEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return HGEMM_OK;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != HGEMM_OK) return rc;
  cudaError_t e;
  // Row chunks of A and C pipeline the copies with the product: chunk i's
  // rows of C are computed as soon as its rows of A (and all of B) have
  // landed, while later rows of A are still arriving and earlier rows of C
  // are copied back. Small problems take a single chunk.
  const int64_t bytes = 2 * (M * K + N * K + M * N);
  int64_t chunks = (bytes >= (int64_t{32} << 20) && M >= 2048) ? 8 : 1;
  int64_t rows = (M + chunks - 1) / chunks;
  rows = (rows + 255) / 256 * 256;
  chunks = (M + rows - 1) / rows;
  if (chunks <= 1) {
    if (M * K &&
        (e = cudaMemcpyAsync(dA, hA, 2 * M * K, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
      return cuda_fail(e);
    if (N * K &&
        (e = cudaMemcpyAsync(dB, hB, 2 * N * K, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
      return cuda_fail(e);
    if ((rc = dispatch(dense(dA, dB, dC, M, N, K), kPlainEpilogue, *dev, stream)) != HGEMM_OK) return rc;
    if ((e = cudaMemcpyAsync(hC, dC, 2 * M * N, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
      return cuda_fail(e);
    return HGEMM_OK;
  }
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  if ((rc = pipe_for_current_device(&hp)) != HGEMM_OK) return rc;
  cudaEvent_t* ev = hp->ev;
  // everything starts after the work already on `stream`
  if ((e = cudaEventRecord(ev[0], stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->in, ev[0], 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->out, ev[0], 0)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaMemcpyAsync(dB, hB, 2 * N * K, cudaMemcpyHostToDevice, hp->in)) != cudaSuccess)
    return cuda_fail(e);
  for (int64_t i = 0; i < chunks; ++i) {
    const int64_t r0 = i * rows;
    const int64_t mi = (M - r0 < rows) ? M - r0 : rows;
    cudaEvent_t in_done = ev[2 + 2 * i], prod_done = ev[3 + 2 * i];
    if (K && (e = cudaMemcpyAsync(dA + r0 * K, hA + r0 * K, 2 * mi * K, cudaMemcpyHostToDevice,
                                  hp->in)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaEventRecord(in_done, hp->in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, in_done, 0)) != cudaSuccess)
      return cuda_fail(e);
    if ((rc = dispatch(dense(dA + r0 * K, dB, dC + r0 * N, mi, N, K), kPlainEpilogue, *dev, stream)) !=
        HGEMM_OK)
      return rc;
    if ((e = cudaEventRecord(prod_done, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->out, prod_done, 0)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaMemcpyAsync(hC + r0 * N, dC + r0 * N, 2 * mi * N, cudaMemcpyDeviceToHost,
                             hp->out)) != cudaSuccess)
      return cuda_fail(e);
  }
  // `stream` completes only after the last copy back
  if ((e = cudaEventRecord(ev[1], hp->out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, ev[1], 0)) != cudaSuccess)
    return cuda_fail(e);
  return HGEMM_OK;
}

int hgemm_select_path(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K) {
  const Gemm g = dense(A, B, const_cast<void*>(C), M, N, K);
  int rc = validate(g);
  if (rc != HGEMM_OK) return rc;
  int split = 1, tile_n = hg::kPairBN;
  return choose_path(g, *g_last_profile.load(std::memory_order_acquire), false, &split, &tile_n);
}

int hgemm_force_split(int split, int tile_n) {
  const bool ok = (split == 0 && tile_n == 0) || (split == 2 && tile_n == 128) ||
                  (tile_n == 256 && split >= 2 && split <= 4);
  if (!ok) return HGEMM_ERR_INVALID_ARG;
  g_forced_split.store(split * 1024 + tile_n);
  return HGEMM_OK;
}

int hgemm_force_trsm_schedule(int schedule) {
  if (schedule != HGEMM_TRSM_AUTO && schedule != HGEMM_TRSM_RECURSIVE && schedule != HGEMM_TRSM_CHAIN &&
      schedule != HGEMM_TRSM_CHAIN_FUSED && schedule != HGEMM_TRSM_CHAIN_SPLIT)
    return HGEMM_ERR_INVALID_ARG;
  g_trsm_schedule.store(schedule);
  return HGEMM_OK;
}

int hgemm_trsm_last_schedule(void) { return t_trsm_schedule; }

int hgemm_force_path(int path) {
  if (path != -1 && path != HGEMM_PATH_TC && path != HGEMM_PATH_TC_NARROW && path != HGEMM_PATH_TC_PAIR &&
      path != HGEMM_PATH_TC_WIDE && path != HGEMM_PATH_SKINNY && path != HGEMM_PATH_GENERIC)
    return HGEMM_ERR_INVALID_ARG;
  g_forced_path.store(path);
  return HGEMM_OK;
}

int hgemm_device_status(cudaStream_t stream) {
  DeviceState* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != HGEMM_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  if ((e = cudaMemcpy(&word, t_ctx.status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e);
  const int zero = 0;
  // the debug build's check words: a failed check outranks the timeout it
  // may have caused (a skipped copy leaves a barrier short)
  int check = 0;
  for (int* w : t_ctx.debug) {
    if (!w) continue;
    int v = 0;
    if ((e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
      if (check == 0) check = v;
      if ((e = cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e);
    }
  }
  if (word != 0) {
    if ((e = cudaMemcpy(t_ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e);
  }
  if (check != 0) {
    t_debug_code = check;
    return HGEMM_ERR_DEBUG_CHECK;
  }
  return word != 0 ? HGEMM_ERR_TIMEOUT : HGEMM_OK;
}

int hgemm_debug_code(void) { return t_debug_code; }

int hgemm_debug_build(void) {
#ifdef HGEMM_DEBUG
  return 1;
#else
  return 0;
#endif
}

int hgemm_debug_selftest(void) {
  // The predicates of the device checks on values inside and just outside
  // their ranges (never run on a GPU with bad values). Bit i set: case i wrong.
  int bad = 0, i = 0;
  auto expect = [&](bool got, bool want) {
    if (got != want) bad |= 1 << i;
    ++i;
  };
  expect(hg::dbg_range_ok(1024, 16, 1024, 4096), true);
  expect(hg::dbg_range_ok(1024 + 4096 - 16, 16, 1024, 4096), true);
  expect(hg::dbg_range_ok(1024 + 4096 - 8, 16, 1024, 4096), false);   // runs past the end
  expect(hg::dbg_range_ok(1016, 16, 1024, 4096), false);              // starts in the reserved part
  expect(hg::dbg_range_ok(0xFFFFFFF0u, 32, 1024, 4096), false);       // wraps around
  expect(hg::dbg_range_ok(1024, 8192, 1024, 4096), false);            // larger than the window
  expect(hg::dbg_tma_x_ok(64, 2), true);
  expect(hg::dbg_tma_x_ok(8, 2), true);
  expect(hg::dbg_tma_x_ok(4, 2), false);                              // 8 bytes: not a multiple of 16
  expect(hg::dbg_tma_x_ok(-8, 2), true);                              // negative but aligned
  expect(hg::dbg_tma_x_ok(-3, 2), false);
  expect(hg::dbg_tmem_ok((127u << 16) | 480u, 32), true);
  expect(hg::dbg_tmem_ok(481u, 32), false);                           // past column 511
  expect(hg::dbg_tmem_ok(128u << 16, 32), false);                     // past lane 127
  expect(hg::dbg_index_ok(0, 1), true);
  expect(hg::dbg_index_ok(1, 1), false);
  expect(hg::dbg_index_ok(-1, 5), false);
  expect(hg::dbg_aligned(4096, 16), true);
  expect(hg::dbg_aligned(4104, 16), false);
  return bad;
}

int hgemm_launch_floor(int pair_config, cudaStream_t stream) {
  DeviceState* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != HGEMM_OK) return rc;
  const cudaError_t e = hg::launch_floor(pair_config, dev->num_sms, hg::pair_smem_bytes(), stream);
  return e == cudaSuccess ? HGEMM_OK : cuda_fail(e);
}

int hgemm_set_wait_timeout(unsigned long long ns) {
  g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs);
  return HGEMM_OK;
}

int hgemm_debug_inject(int what) {
  if (what != HGEMM_INJECT_NONE && what != HGEMM_INJECT_DROP_ARRIVAL) return HGEMM_ERR_INVALID_ARG;
  g_inject.store(what);
  return HGEMM_OK;
}

int hgemm_last_cuda_error(void) { return t_last_cuda_error; }

const char* hgemm_status_string(int status) {
  switch (status) {
    case HGEMM_OK:
      return "ok";
    case HGEMM_ERR_INVALID_ARG:
      return "invalid argument (dimension out of range or NULL pointer)";
    case HGEMM_ERR_ALIAS:
      return "C overlaps A or B";
    case HGEMM_ERR_UNSUPPORTED_DEVICE:
      return "current device is not an sm_103 (GB300) GPU";
    case HGEMM_ERR_CUDA:
      return "a CUDA call failed (see hgemm_last_cuda_error)";
    case HGEMM_ERR_TIMEOUT:
      return "a kernel wait timed out; the output is incomplete";
    case HGEMM_ERR_DEBUG_CHECK:
      return "a device-side check of the debug build failed (see hgemm_debug_code); the output is incomplete";
    default:
      return "unknown status";
  }
}

int hgemm_version(void) { return (0 << 16) | 1; }

}  // extern "C"
