/*
 * hgemm.h — C ABI of the GB300 (sm_103a) FP16 tensor-core GEMM, C = A·B.
 *
 * The operation, as stated in "Nvidia Tensor Core-MMA PTX编程入门", §4 示例:
 * C = A·B with A an M×K row-major matrix, B a K×N column-major matrix and C
 * an M×N row-major matrix, all IEEE binary16 (FP16). In memory:
 *
 *     A(i, k) = A[i*K + k]      0 <= i < M, 0 <= k < K
 *     B(k, j) = B[j*K + k]      0 <= j < N   (each column of B is contiguous)
 *     C(i, j) = C[i*N + j]
 *
 * Products are accumulated in FP32 ("GPU架构与CUDA", 混合精度核函数: FP16 × FP16
 * accumulated in FP32) and each output is rounded once to FP16, round to
 * nearest even. C is overwritten; there is no alpha, beta or accumulation
 * into C. Terms outside the matrices contribute nothing and nothing outside
 * the M×N region of C is written ("GPU架构与CUDA", 共享内存与分块: zero-filled
 * tile loads and a guarded store).
 *
 * Element type: FP16 values are passed as their 16-bit patterns
 * (hgemm_half_t); __half, torch.float16 and numpy.float16 share the layout.
 *
 * Streams ("GPU架构与CUDA", 流与并发): every entry point that computes only
 * enqueues work on the caller's stream and returns; results are ready once
 * the stream has been synchronised. Nothing here synchronises unless its
 * comment says so.
 *
 * Ownership: the caller allocates, owns and frees every buffer. The library
 * allocates no device memory and keeps no pointer after a call returns.
 * Inputs must not be written while the enqueued work runs.
 *
 * Errors: every int-returning call returns HGEMM_OK (0) or a negative status
 * below. A failing call enqueues nothing. After HGEMM_ERR_CUDA, the CUDA
 * error that caused it is returned by hgemm_last_cuda_error() on the same
 * host thread.
 *
 * Device: the kernels are built for sm_103a only (GB300). On any other device
 * the computing calls return HGEMM_ERR_UNSUPPORTED_DEVICE; there is no
 * fallback path of any kind.
 */
#ifndef HGEMM_H_
#define HGEMM_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define HGEMM_API __attribute__((visibility("default")))
#else
#define HGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t hgemm_half_t; /* IEEE binary16 bit pattern */

/* status codes */
#define HGEMM_OK 0
#define HGEMM_ERR_INVALID_ARG (-1)        /* bad dimension, NULL or odd pointer */
#define HGEMM_ERR_ALIAS (-2)              /* C overlaps A or B */
#define HGEMM_ERR_UNSUPPORTED_DEVICE (-3) /* current device is not compute capability 10.3 */
#define HGEMM_ERR_CUDA (-4)               /* a CUDA runtime/driver call failed (see hgemm_last_cuda_error) */
#define HGEMM_ERR_TIMEOUT (-5)            /* a kernel's bounded wait gave up (see hgemm_device_status) */
#define HGEMM_ERR_DEBUG_CHECK (-6)        /* a device-side check of the -DHGEMM_DEBUG build failed */

/* kernel paths, as reported by hgemm_select_path */
#define HGEMM_PATH_NONE 0     /* M == 0 or N == 0: nothing to do */
#define HGEMM_PATH_ZERO 1     /* K == 0: C is filled with +0 (the empty sum; hgemm_ex: f(beta·C + bias)) */
#define HGEMM_PATH_TC 2       /* tcgen05 + TMA persistent kernel, one CTA per 128×256 tile */
#define HGEMM_PATH_SKINNY 3   /* tcgen05 + TMA kernel for small N, split over K */
#define HGEMM_PATH_GENERIC 4  /* tcgen05 kernel fed by plain loads: any alignment */
#define HGEMM_PATH_TC_PAIR 5  /* tcgen05 + TMA persistent kernel, CTA pairs per 256×256 tile */
#define HGEMM_PATH_TC_WIDE 6  /* tcgen05 + TMA persistent kernel, CTA pairs per 256×512 tile */
#define HGEMM_PATH_TC_NARROW 7 /* the HGEMM_PATH_TC kernel on 128×64 tiles: outputs one wave covers */

/* Largest M, N or K accepted (TMA coordinates are signed 32-bit). */
#define HGEMM_MAX_DIM ((int64_t)0x7FFFFFFF)
#define HGEMM_TRMM_MAX_N 16384          /* largest triangle hgemm_trmm accepts */

/*
 * hgemm — C = A·B on `stream` (see the top of this file for layouts).
 *
 *   A, B, C  device pointers (or managed memory visible to the current
 *            device), each at least 2-byte aligned (FP16 elements). When A,
 *            B, C are 16-byte aligned and K and N are multiples of 8 the
 *            TMA-fed kernels run; otherwise a tensor-core kernel fed by plain
 *            loads does the same arithmetic.
 *   M, N, K  0 <= M, N, K <= HGEMM_MAX_DIM. M == 0 or N == 0 is a no-op;
 *            K == 0 sets every C(i, j) to +0. A and B may be NULL when their
 *            size is 0, C when M*N == 0.
 *   stream   CUDA stream of the current device (0 = legacy default stream).
 *
 * Returns HGEMM_OK once the work is enqueued, else an error status and
 * nothing is enqueued: HGEMM_ERR_INVALID_ARG, HGEMM_ERR_ALIAS (the bytes of C
 * overlap those of A or B), HGEMM_ERR_UNSUPPORTED_DEVICE, HGEMM_ERR_CUDA
 * (launch or tensor-map encoding failure).
 */
HGEMM_API int hgemm(const hgemm_half_t *A, const hgemm_half_t *B, hgemm_half_t *C,
          int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * hgemm_ex — the fused product of "GPU架构与CUDA", 核函数融合 (matmul, bias
 * add and ReLU in one kernel: the intermediate never goes to memory), with
 * BLAS-style scaling:
 *
 *   C[i·N + j] = fp16_rne( f( alpha · Σ_k A[i·K + k] · B[j·K + k]
 *                             + beta · C_old[i·N + j] + bias[j] ) )
 *
 * f is max(·, 0) when relu != 0, else the identity; bias holds N FP16 values,
 * one per column of C (an output feature of the page's matmul(x, W) + bias),
 * or is NULL. The sum accumulates in FP32 on the tensor cores and the
 * epilogue arithmetic is FP32, rounded once to FP16. When beta == 0, C is
 * not read (a NaN there does not propagate); otherwise C is read and
 * overwritten in place. Layouts, sizes, streams and ownership as for hgemm;
 * bias must be 2-byte aligned and must not overlap C (HGEMM_ERR_ALIAS).
 * hgemm(A, B, C, M, N, K, s) is hgemm_ex(A, B, C, M, N, K, 1, 0, NULL, 0, s).
 * K = 0 gives C := f(beta · C_old + bias). Same return values as hgemm.
 */
HGEMM_API int hgemm_ex(const hgemm_half_t *A, const hgemm_half_t *B, hgemm_half_t *C,
             int64_t M, int64_t N, int64_t K, float alpha, float beta,
             const hgemm_half_t *bias, int relu, cudaStream_t stream);

/*
 * hgemm_strided — hgemm_ex on sub-matrices, the form the recursive TRMM of
 * "异构计算中高性能TRMM与TRSM的递归算法实现" (§2.1 blocking, §2.2 the GEMM
 * update of an off-diagonal block) needs: row pitches in elements, with
 * A(i,k) at A[i·lda + k], B(k,j) at B[j·ldb + k] (column j of B still
 * contiguous) and C(i,j) at C[i·ldc + j]; lda ≥ K, ldb ≥ K, ldc ≥ N.
 * The tensor-core paths need 16-byte-aligned base addresses, pitches that
 * are multiples of 8 and N a multiple of 8; anything else takes
 * HGEMM_PATH_GENERIC. The span C occupies must not overlap the spans of A, B
 * or bias (HGEMM_ERR_ALIAS). hgemm_ex(...) is hgemm_strided with lda = ldb = K
 * and ldc = N. Same return values as hgemm.
 */
HGEMM_API int hgemm_strided(const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
                  hgemm_half_t *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                  float alpha, float beta, const hgemm_half_t *bias, int relu,
                  cudaStream_t stream);

/*
 * hgemm_layout — hgemm_strided with a storage order chosen per operand, the
 * other layouts of the product (the CUDA chapter of "GPU架构与CUDA",
 * 共享内存与分块, stores B row-major, K×N with N contiguous):
 *
 *   a_layout  HGEMM_A_ROW_MAJOR: A(i,k) at A[i·lda + k], lda ≥ K (as hgemm);
 *             HGEMM_A_COL_MAJOR: A(i,k) at A[k·lda + i], lda ≥ M;
 *   b_layout  HGEMM_B_COL_MAJOR: B(k,j) at B[j·ldb + k], ldb ≥ K (as hgemm);
 *             HGEMM_B_ROW_MAJOR: B(k,j) at B[k·ldb + j], ldb ≥ N;
 *
 * C(i,j) at C[i·ldc + j] always. Same epilogue (alpha, beta, bias, relu),
 * ownership, alias and error rules as hgemm_ex; an unknown layout value is
 * HGEMM_ERR_INVALID_ARG. Operands that TMA can describe (16-byte aligned
 * bases and pitches, N a multiple of 8) take the tensor-core path hgemm
 * would take for the shape (the pair kernel where that is the single-CTA
 * one), reading an M- or N-contiguous operand as MN-major tiles; the others
 * go to the generic kernel, which gathers them.
 */
#define HGEMM_A_ROW_MAJOR 0
#define HGEMM_A_COL_MAJOR 1
#define HGEMM_B_COL_MAJOR 0
#define HGEMM_B_ROW_MAJOR 1
HGEMM_API int hgemm_layout(int a_layout, int b_layout, const hgemm_half_t *A, int64_t lda,
                 const hgemm_half_t *B, int64_t ldb, hgemm_half_t *C, int64_t ldc, int64_t M,
                 int64_t N, int64_t K, float alpha, float beta, const hgemm_half_t *bias,
                 int relu, cudaStream_t stream);

/*
 * hgemm_trmm — the triangular product of "异构计算中高性能TRMM与TRSM的递归算法实现"
 * §2.2 (left side, lower triangle, transposed: B ← alpha·Aᵀ·B), out of place:
 *
 *     C = alpha · Aᵀ · B
 *
 * A is n×n lower triangular and only its lower triangle (row ≥ column) is
 * used: the entries above the diagonal may hold anything, NaN included (they
 * lie inside A's span and may be loaded, never used); B and C are n×m. All three are column-major, as on the page (Julia):
 * A(r,c) at A[c·lda + r], B(r,j) at B[j·ldb + r], C(r,j) at C[j·ldc + r],
 * with lda, ldb, ldc ≥ n; n ≤ HGEMM_TRMM_MAX_N (n or m = 0: nothing to do). By the page's
 * recursion (§2.1, §2.2): a block splits into halves; C1 = A11ᵀ·B1, then the
 * GEMM update C1 += A21ᵀ·B2 (hgemm's accumulate epilogue), then C2 = A22ᵀ·B2;
 * blocks of order ≤ 256 (the page's threshold) are leaves, all computed by
 * one launch of masked products, which also carries the updates of at most
 * 2^33 multiply-adds (m·s1·s2) when n is a multiple of 64: a leaf's product
 * then runs on over those updates' columns of A and B (the same sum, one FP16
 * rounding fewer). Storage is FP16 (each update rounds its block once),
 * accumulation FP32 within each product. C must not overlap A
 * or B (HGEMM_ERR_ALIAS); the calls are enqueued on `stream`. Same return
 * values as hgemm.
 */
HGEMM_API int hgemm_trmm(const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
               hgemm_half_t *C, int64_t ldc, int64_t n, int64_t m, float alpha,
               cudaStream_t stream);

/*
 * hgemm_trsm — the triangular solve of "异构计算中高性能TRMM与TRSM的递归算法实现"
 * §2.3, in the variant of hgemm_trmm's product (left side, lower triangle,
 * transposed):
 *
 *     solve  Aᵀ · X = alpha · B  for X
 *
 * A is n×n lower triangular and only its lower triangle (row ≥ column) is
 * used: the entries above the diagonal may hold anything, NaN included (they
 * lie inside A's span and may be loaded, never used); B and X are n×m (m
 * right-hand sides). All three are column-major:
 * A(r,c) at A[c·lda + r], B(r,j) at B[j·ldb + r], X(r,j) at X[j·ldx + r],
 * with lda, ldb, ldx ≥ n (n or m = 0: nothing to do). X = B with ldx = ldb
 * solves in place (B is overwritten, as in BLAS); any other overlap of X with
 * A or B is HGEMM_ERR_ALIAS. By the page's recursion (§2.1): X := alpha·B;
 * a block splits into halves, the second is solved first, then the GEMM
 * update X1 -= A21ᵀ·X2 (hgemm's accumulate epilogue with alpha = -1), then
 * the first half; diagonal blocks of order ≤ 256 are solved by substitution,
 * the right-hand sides spread over thread blocks (§2.3; the page puts a
 * barrier after every row, this kernel one per group of 32 rows). Storage is FP16 (X is rounded after the scaling, after each update
 * and after each diagonal solve), arithmetic FP32. A zero on the diagonal is
 * not reported: as in BLAS, the result then holds Inf or NaN. The calls are
 * enqueued on `stream`, one after another. Same return values as hgemm.
 */
HGEMM_API int hgemm_trsm(const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
               hgemm_half_t *X, int64_t ldx, int64_t n, int64_t m, float alpha,
               cudaStream_t stream);

/*
 * hgemm_trsm_workspace_size — bytes of device workspace hgemm_trsm_ws uses
 * for a triangle of order n: 512 KiB per diagonal block of order ≤ 512 of
 * the recursion, plus, for the one-launch schedule, one spare block of 512
 * KiB and 4 KiB of synchronisation words (n = 8192: 16 blocks, 8.5 MiB +
 * 4 KiB). 0 for n ≤ 0 or n beyond 128 such blocks. Pure host logic.
 */
HGEMM_API size_t hgemm_trsm_workspace_size(int64_t n);

/*
 * hgemm_trsm_ws — hgemm_trsm (same system, operands, recursion and return
 * values) with a caller-owned device workspace of at least
 * hgemm_trsm_workspace_size(n) bytes, 16-byte aligned (256 as cudaMalloc
 * gives), not overlapping A, B or X (HGEMM_ERR_ALIAS), not used by any
 * other work until the stream has passed this call. With it, when X is
 * 16-byte aligned with ldx a multiple of 8, the recursion stops at diagonal
 * blocks of order ≤ 512: one launch first computes their inverses (FP32
 * arithmetic, stored FP16 in the workspace), and each is then solved as an
 * in-place tensor-core product X_bᵀ := X_bᵀ · L_b⁻¹ instead of by
 * substitution (a block whose order is not a multiple of 8 still recurses to
 * the substitution kernel). The substitution then happens once per block for
 * the identity rather than per right-hand side, and the deepest updates of
 * the recursion are inside the inverses.
 * Schedule: when m ≤ 1024, the workspace is the full
 * hgemm_trsm_workspace_size(n), A is 16-byte aligned with lda a multiple of
 * 8 and the recursion has at most 16 diagonal blocks (n ≤ 8192),
 * everything after the inverses runs as ONE persistent cooperative launch,
 * one phase per block in the recursion's order with grid-wide barriers
 * between them: phase k solves block k as one product,
 * X_kᵀ := T_kᵀ·L_k⁻¹ − X_{k−1}ᵀ·M_k, where T_k is block k's right-hand side
 * after the updates from the blocks solved up to two before it and
 * M_k = C_k·L_k⁻¹ (C_k the part of A coupling block k−1 to block k,
 * computed one phase ahead into a spare slot of the workspace), and
 * subtracts X_{k−1}'s contribution from every block after k at once (the
 * recursion's update sums, split per block: right-looking). Otherwise (a
 * workspace of only the inverses' size, as earlier versions asked for, or
 * the limits above) the recursion runs as a sequence of launches (products
 * by the inverses, GEMM updates). hgemm_force_trsm_schedule chooses for
 * testing; hgemm_trsm_last_schedule tells which one a call took.
 * Rounding: each solved block is rounded once to FP16, the inverse once
 * more; X is rounded after every update it receives (the recursion: once per
 * level whose first half holds the block; the one launch: once per block
 * solved two or more before it, and M_k once). A null workspace, one too small or not 16-byte
 * aligned is HGEMM_ERR_INVALID_ARG; X not suited to the tensor-core path, or
 * a path forced by hgemm_force_path, solves as hgemm_trsm does.
 * Accuracy against hgemm_trsm: rounding L_b⁻¹ to FP16 adds at most
 * 2^-11·(|L_b⁻¹|ᵀ·|b_b|) to each x in block b (b_b the block's right-hand
 * side after the updates), so the result meets the per-element tolerance
 * 1e-2·max(1, |x|) wherever |L_b⁻¹|ᵀ·|b_b| <= 16·max(1, |x_b|), i.e. while
 * the diagonal blocks' inverses do not cancel heavily. Measured against the
 * FP64 solve: with a diagonal in [1, 2) and a strict lower part below c/n,
 * both entry points stay within that tolerance up to c = 512 at n = 4096
 * and 8192 (entries up to 1/8 and 1/16) and up to c = 256 at n = 1024
 * (entries up to 1/4); past that (n = 1024, c = 512: the solution grows to
 * ~350 from a right-hand side below 1) neither does, while the
 * componentwise backward error |Aᵀ·X − alpha·B| / (|Aᵀ|·|X| + |alpha·B|)
 * of both stays below 4·2^-11.
 */
HGEMM_API int hgemm_trsm_ws(const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
                  hgemm_half_t *X, int64_t ldx, int64_t n, int64_t m, float alpha,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * hgemm_trsm_op — the triangular solve in either orientation, with or
 * without a workspace:
 *
 *     op = HGEMM_OP_N:  solve  A · X = alpha · B   (the page's literal reading
 *                                                    of §2.3, X = A\B column by
 *                                                    column)
 *     op = HGEMM_OP_T:  solve  Aᵀ · X = alpha · B  (hgemm_trsm's system)
 *
 * Same operands as hgemm_trsm: A n×n lower triangular (only row ≥ column is
 * used), B and X n×m, all column-major with pitches ≥ n; X = B with ldx = ldb
 * solves in place; any other overlap is HGEMM_ERR_ALIAS. With op =
 * HGEMM_OP_N the recursion (§2.1) runs the other way round: a block's first
 * half is solved first, then the GEMM update X2 -= A21·X1 (hgemm_layout's
 * N-contiguous second operand: row k of A21ᵀ is a piece of column k of A),
 * then the second half; diagonal blocks of order ≤ 256 are solved by forward
 * substitution with the right-hand sides spread over thread blocks, like
 * hgemm_trsm's. workspace may be null (workspace_bytes then 0) to solve
 * every diagonal block by substitution, as hgemm_trsm does; otherwise it is
 * hgemm_trsm_ws's workspace (same size, alignment and rules) and the blocks
 * of order ≤ 512 are solved through their inverses, the same inverses for
 * both orientations (op = N multiplies X_bᵀ by L_b⁻ᵀ, op = T by L_b⁻¹).
 * Storage, rounding and accuracy as hgemm_trsm and hgemm_trsm_ws. An op
 * other than the two, or a null workspace with a nonzero size, is
 * HGEMM_ERR_INVALID_ARG; otherwise the same return values as hgemm_trsm_ws.
 */
#define HGEMM_OP_N 0
#define HGEMM_OP_T 1
HGEMM_API int hgemm_trsm_op(int op, const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
                  hgemm_half_t *X, int64_t ldx, int64_t n, int64_t m, float alpha,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * TRSM schedules (hgemm_trsm_last_schedule, hgemm_force_trsm_schedule):
 * SUBSTITUTION: no workspace (or X not suited to it): the recursion's
 * launches with every diagonal block of order ≤ 256 solved by substitution;
 * RECURSIVE: the recursion's launches, blocks of order ≤ 512 solved by
 * their inverses; CHAIN: the inverses' launch, then one persistent launch
 * (hgemm_trsm_ws), in one of two plans: CHAIN_FUSED, one phase per block
 * (its product folds in the update from the block before through M_k),
 * or CHAIN_SPLIT, two phases per block (the product by the inverse, then
 * the update of every later block); the library takes the plan its cost
 * model of the two finds faster (fused for few right-hand sides).
 */
#define HGEMM_TRSM_AUTO 0
#define HGEMM_TRSM_SUBSTITUTION 1
#define HGEMM_TRSM_RECURSIVE 2
#define HGEMM_TRSM_CHAIN 3
#define HGEMM_TRSM_CHAIN_FUSED 4
#define HGEMM_TRSM_CHAIN_SPLIT 5

/*
 * hgemm_force_trsm_schedule — testing and profiling aid: HGEMM_TRSM_RECURSIVE
 * keeps later solves with a workspace on the recursion's launches;
 * HGEMM_TRSM_CHAIN takes the one-launch schedule wherever it can run (also
 * past m = 1024, where it is slower: its product phases must fit one wave
 * of tiles, m up to ~9,700; n ≤ 8192) with the plan of the library's
 * choice, HGEMM_TRSM_CHAIN_FUSED or HGEMM_TRSM_CHAIN_SPLIT with that plan;
 * HGEMM_TRSM_AUTO (the default) chooses as hgemm_trsm_ws describes.
 * Returns HGEMM_OK, or HGEMM_ERR_INVALID_ARG for another value.
 * Process-wide, like hgemm_force_path.
 */
HGEMM_API int hgemm_force_trsm_schedule(int schedule);

/*
 * hgemm_trsm_last_schedule — the HGEMM_TRSM_* schedule of the last
 * triangular solve enqueued on this host thread (0 before any; a chain
 * reports its plan, HGEMM_TRSM_CHAIN_FUSED or HGEMM_TRSM_CHAIN_SPLIT). Host
 * logic.
 */
HGEMM_API int hgemm_trsm_last_schedule(void);

/*
 * hgemm_trsm_noalloc — hgemm_trsm_ws for callers that cannot allocate device
 * memory: code whose device memory all belongs to another allocator (a
 * framework's caching pool, a fixed budget reserved up front) and which may
 * not call cudaMalloc itself, or which must not pay cudaMalloc's implicit
 * synchronisation. The pages have no counterpart of this entry point; it is
 * an addition for such callers.
 *
 * Same system, operands, results and return values as hgemm_trsm_ws, whose
 * workspace here is a fixed array of HGEMM_TRSM_NOALLOC_MAX_BYTES (8.5 MiB +
 * 4 KiB) inside the library, present on every device that loads the library until
 * the process exits. Nothing is allocated: no cudaMalloc or cudaFree, no
 * allocating library call. Limit: triangles whose recursion has at most 16
 * diagonal blocks of order ≤ 512, which is every n ≤ 8192; a larger n
 * (hgemm_trsm_workspace_size(n) > HGEMM_TRSM_NOALLOC_MAX_BYTES) returns
 * HGEMM_ERR_INVALID_ARG and enqueues nothing.
 *
 * The device check comes first: on a device other than an sm_103 GPU the
 * call returns HGEMM_ERR_UNSUPPORTED_DEVICE, like hgemm_trsm_ws. The first
 * call on a host thread in a given CUDA context (the device's primary context
 * as the runtime makes it current) looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it for that
 * thread and context; a call in another context, or after the primary context
 * was recreated by a device reset, looks it up again. Make each host thread's
 * first call before any stream capture on the device. Every call on a device
 * shares the one array, which keeps the last call's contents (each call
 * writes every entry it reads, so nothing needs clearing): calls whose work
 * overlaps on the GPU (other streams, other host threads) race on it and
 * must be ordered by the caller, e.g. issued on one stream.
 */
#define HGEMM_TRSM_NOALLOC_MAX_BYTES ((17u << 19) + 4096u)
HGEMM_API int hgemm_trsm_noalloc(const hgemm_half_t *A, int64_t lda, const hgemm_half_t *B, int64_t ldb,
                       hgemm_half_t *X, int64_t ldx, int64_t n, int64_t m, float alpha,
                       cudaStream_t stream);

/*
 * hgemm_host — the same product for operands held in HOST memory.
 *
 * Copies hA -> dA (M*K values) and hB -> dB (N*K values), computes
 * C = A·B into dC (same rules as hgemm) and copies dC -> hC (M*N values).
 * All of it happens after the work already enqueued on `stream`, and
 * `stream` completes only after the last copy back. For problems of 32 MB
 * or more with M >= 2048 the work is pipelined over row chunks: B is copied
 * first, then chunk i's rows of A are copied on a helper stream while the
 * product of the previous chunk runs on `stream` and a second helper stream
 * copies finished rows of C back (helper streams and events are created once
 * per device and kept; no device memory is allocated). The caller provides
 * and owns every buffer. Host buffers should be page-locked for the copies
 * to be asynchronous; hC is valid once `stream` has been synchronised. Same
 * return values as hgemm.
 */
HGEMM_API int hgemm_host(const hgemm_half_t *hA, const hgemm_half_t *hB, hgemm_half_t *hC,
               int64_t M, int64_t N, int64_t K,
               hgemm_half_t *dA, hgemm_half_t *dB, hgemm_half_t *dC,
               cudaStream_t stream);

/*
 * hgemm_select_path — the HGEMM_PATH_* that hgemm would run for these
 * arguments on a GB300, or a negative status for invalid arguments. Pure
 * host logic: touches no device and needs no GPU. Honours hgemm_force_path.
 * hgemm_ex with a fused epilogue takes the same path, except that it takes
 * HGEMM_PATH_TC_PAIR where this reports HGEMM_PATH_TC_WIDE.
 */
HGEMM_API int hgemm_select_path(const void *A, const void *B, const void *C,
                      int64_t M, int64_t N, int64_t K);

/*
 * hgemm_force_path — overrides path selection for later calls in this
 * process (testing and profiling). `path` is HGEMM_PATH_TC,
 * HGEMM_PATH_TC_NARROW, HGEMM_PATH_TC_PAIR, HGEMM_PATH_TC_WIDE,
 * HGEMM_PATH_SKINNY or HGEMM_PATH_GENERIC, or -1 to
 * restore automatic selection. A forced TMA path still falls back to GENERIC
 * when the operands are not aligned for TMA. In hgemm_trmm a forced path runs
 * every off-diagonal update as a product of its own (none is carried by the
 * leaves; HGEMM_PATH_GENERIC also computes the leaves on the generic
 * kernel); in hgemm_trsm_ws it solves the diagonal blocks by substitution.
 * Returns HGEMM_OK or HGEMM_ERR_INVALID_ARG.
 *
 * Tuning overrides read once per process from the environment:
 * HGEMM_GROUP_M (a positive integer) sets how many M-tiles the tensor-core
 * kernels' grouped raster order keeps together (default 12);
 * HGEMM_TAIL_SPLIT=0 keeps whole 256×256 tiles in the last, partly filled
 * wave of the CTA-pair kernel instead of cutting them into 128- or
 * 64-column parts.
 */
HGEMM_API int hgemm_force_path(int path);

/*
 * hgemm_force_split — testing aid for the split-K path (HGEMM_PATH_SKINNY):
 * later calls that take that path use `split` K-slices over tiles `tile_n`
 * columns wide, when that configuration's clusters fit on the device at once
 * and K has at least `split` blocks of 64 (otherwise the automatic choice
 * stands). Configurations: (2, 128), (2, 256), (3, 256), (4, 256); (0, 0)
 * restores the automatic choice. Returns HGEMM_OK or HGEMM_ERR_INVALID_ARG.
 * Pure host state, process-wide.
 */
HGEMM_API int hgemm_force_split(int split, int tile_n);

/*
 * hgemm_device_status — synchronises `stream`, then reads and clears the
 * library's device watchdog word on the current device. Every wait inside the
 * kernels is bounded in time; a wait that gives up records itself there and
 * its kernel returns early, leaving C incomplete. Returns HGEMM_OK,
 * HGEMM_ERR_TIMEOUT, HGEMM_ERR_DEBUG_CHECK (debug build: a device-side check
 * failed; it outranks a timeout the skipped access caused), or
 * HGEMM_ERR_CUDA if the synchronisation failed.
 */
HGEMM_API int hgemm_device_status(cudaStream_t stream);

/*
 * hgemm_set_wait_timeout — time limit, in nanoseconds, of every wait inside
 * the kernels of later calls in this process (0 restores the default, 2 s).
 * Returns HGEMM_OK.
 */
HGEMM_API int hgemm_set_wait_timeout(unsigned long long ns);

/* fault injection for testing the watchdog */
#define HGEMM_INJECT_NONE 0
#define HGEMM_INJECT_DROP_ARRIVAL 1 /* producer withholds its first stage's arrival */

/*
 * hgemm_debug_inject — testing aid for the watchdog. With
 * HGEMM_INJECT_DROP_ARRIVAL, the TMA producer of the tensor-core kernels of
 * later calls withholds the barrier arrival of its first stage (its copies
 * are still issued and land), so the MMA issuer's bounded wait gives up: the
 * kernel records HGEMM_ERR_TIMEOUT in the watchdog word, drains, frees TMEM
 * and returns with C incomplete. No GPU fault is raised and the context
 * stays usable. HGEMM_INJECT_NONE turns it off. Returns HGEMM_OK or
 * HGEMM_ERR_INVALID_ARG.
 */
HGEMM_API int hgemm_debug_inject(int what);

/* hgemm_last_cuda_error — the cudaError_t behind the last HGEMM_ERR_CUDA
 * returned on this host thread (0 if none). */
HGEMM_API int hgemm_last_cuda_error(void);

/*
 * hgemm_launch_floor — measurement aid: enqueues a kernel that does nothing,
 * so that a caller can time the fixed cost of one launch on its GPU and
 * stream (the part of a small product's time that no kernel design
 * removes). pair_config = 0: one CTA of one warp; otherwise the launch
 * configuration of the CTA-pair product kernel (one CTA per SM in clusters
 * of two, 192 threads, the pair kernel's dynamic shared memory,
 * programmatic stream serialization). Touches no memory. Same return values
 * as hgemm (HGEMM_ERR_UNSUPPORTED_DEVICE, HGEMM_ERR_CUDA).
 */
HGEMM_API int hgemm_launch_floor(int pair_config, cudaStream_t stream);

/*
 * The -DHGEMM_DEBUG build (tensor_core_dense_fp16_gb300/build.py --debug:
 * _build/debug/libhgemm.so, loaded when HGEMM_LIBRARY_VARIANT=debug). Its
 * kernels check every shared-memory address a barrier, TMA copy, bulk or
 * asynchronous copy, or ldmatrix uses against the CTA's own shared memory,
 * every TMA innermost coordinate for 16-byte alignment, every TMEM load
 * against lanes 0..127 and columns 0..511, and the global indices and
 * vector alignments of the kernels that address memory themselves. A failed
 * check records a code and skips the access (no trap); hgemm_device_status
 * then returns HGEMM_ERR_DEBUG_CHECK and clears it, and hgemm_debug_code
 * returns the code (101 shared-memory range, 102 TMA coordinate, 103 TMEM
 * range, 104 global index, 105 alignment). The release build has no checks.
 *
 * hgemm_debug_build — 1 in the debug build, 0 otherwise.
 * hgemm_debug_code — the code behind this thread's last HGEMM_ERR_DEBUG_CHECK.
 * hgemm_debug_selftest — host-only: evaluates the checks' predicates on
 *   values inside and just outside their ranges; 0 when every case is
 *   decided correctly, else a bit per wrong case. Needs no GPU.
 */
HGEMM_API int hgemm_debug_build(void);
HGEMM_API int hgemm_debug_code(void);
HGEMM_API int hgemm_debug_selftest(void);

/* hgemm_status_string — static text for a status code; never NULL. */
HGEMM_API const char *hgemm_status_string(int status);

/* hgemm_version — (major << 16) | minor of this library. */
HGEMM_API int hgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HGEMM_H_ */
