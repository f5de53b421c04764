/*
 * The oracle for the FP16 HGEMM C = A·B. TEST INFRASTRUCTURE ONLY: the
 * tests, the smoke check and the benchmark's CPU-baseline leg are the only
 * code allowed to load it. It shares no code, header or table with the CUDA
 * path in tensor_core_dense_fp16_gb300/.
 *
 * What it computes (the plain definition; no blocking, no reordering):
 *
 *     C[i*N + j] = fp16_rne( sum_{k=0}^{K-1} (double)A[i*K + k] * (double)B[j*K + k] )
 *
 *  - Problem and layouts: "Nvidia Tensor Core-MMA PTX编程入门", §4 示例 — A is
 *    M×K row-major, B is K×N column-major (column j is K contiguous values),
 *    C is M×N row-major, all FP16.
 *  - Products of FP16 values, summed at higher precision than FP16:
 *    "GPU架构与CUDA", 混合精度核函数 (FP16 × FP16 accumulated in FP32). The
 *    oracle sums in FP64, which is at least as precise: every FP16×FP16
 *    product is exact in FP64 (11 + 11 significand bits fit in 53), and the
 *    sum runs in increasing k.
 *  - Terms outside the matrix contribute nothing and nothing outside C is
 *    written: "GPU架构与CUDA", 共享内存与分块 (zero-filled tile loads, the
 *    guarded store). Here that is simply the loop bounds.
 *  - The pages do not state how the accumulator becomes FP16; the reading
 *    taken is one IEEE round-to-nearest-even (overflow to ±Inf).
 *
 * The fused variant (oracle_hgemm_ex) follows "GPU架构与CUDA", 核函数融合:
 * the product, a bias add and a ReLU in one pass, the intermediate never
 * leaving the pass. With the BLAS scaling the pages leave open:
 *
 *     C[i*N + j] = fp16_rne( f( alpha * S + beta * C_old[i*N + j] + bias[j] ) )
 *
 * where S is the FP64 sum above, bias (length N, one value per column of C,
 * i.e. per output feature of the page's matmul(x, W) + bias) may be absent,
 * f is max(·, 0) when relu is set and the identity otherwise, and C_old is
 * not read at all when beta == 0 (so a NaN there does not propagate). All of
 * it in FP64, one rounding at the end.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off (no FMA contraction, so
 * x86-64 and AArch64 hosts produce identical bits).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* ---- FP16 (IEEE binary16) <-> double, written out from the format ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);            /* subnormal: frac · 2^-24 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1.frac) · 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. */
uint16_t oracle_double_to_fp16(double x)
{
    if (isnan(x))
        return 0x7e00;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    /* 65504 is the largest finite value; the midpoint to 2^16 is 65520 and a
     * tie there goes to the even neighbour, 2^16, which overflows. */
    if (a >= 65520.0)
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the grid is multiples of 2^-24; rint rounds to the
         * nearest integer, ties to even (default rounding mode). A result of
         * 1024 is the smallest normal, whose encoding is also 1024. */
        double q = rint(a * ldexp(1.0, 24));
        return sign | (uint16_t)q;
    }
    int e2;
    double f = frexp(a, &e2);      /* a = f · 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                /* a = (2f) · 2^e, 2f in [1, 2) */
    double q = rint(ldexp(f, 11)); /* (2f)·1024, rounded: in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7c00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)q - 1024));
}

/* ---- the contraction ---- */

/* The decoded value of every bit pattern, filled once by
 * oracle_fp16_to_double: a cache of the decode, nothing else. */
static double g_decode[65536];
static pthread_once_t g_decode_once = PTHREAD_ONCE_INIT;

static void fill_decode_table(void)
{
    for (uint32_t h = 0; h < 65536u; ++h)
        g_decode[h] = oracle_fp16_to_double((uint16_t)h);
}

/* One entry, pre-rounding: sum over k in increasing order, in FP64. */
static double dot_f64(const uint16_t *A, const uint16_t *B, int64_t i, int64_t j, int64_t K)
{
    double s = 0.0;
    const uint16_t *a = A + i * K;
    const uint16_t *b = B + j * K;
    for (int64_t k = 0; k < K; ++k)
        s += g_decode[a[k]] * g_decode[b[k]];
    return s;
}

/* The fused epilogue's parameters; `on` == 0 means the plain product. */
struct epilogue {
    int on;
    double alpha, beta;
    const uint16_t *bias;   /* length N, or NULL */
    int relu;
};

/* alpha·s + beta·c_old + bias, then the ReLU, all in FP64 (c_old is the
 * entry's previous FP16 value, looked at only when beta != 0). */
static double apply_epilogue(const struct epilogue *ep, double s, uint16_t c_old, int64_t j)
{
    double v = ep->alpha * s;
    if (ep->beta != 0.0)
        v += ep->beta * g_decode[c_old];
    if (ep->bias)
        v += g_decode[ep->bias[j]];
    if (ep->relu && v < 0.0)
        v = 0.0;
    return v;
}

struct rows_job {
    const uint16_t *A, *B;
    uint16_t *C;     /* FP16 result (and, with a fused epilogue, C_old), or NULL */
    double *S;       /* FP64 pre-rounding sums, or NULL */
    int64_t M, N, K;
    int64_t row_lo, row_hi;
    struct epilogue ep;
};

static void *rows_worker(void *arg)
{
    struct rows_job *jb = (struct rows_job *)arg;
    for (int64_t i = jb->row_lo; i < jb->row_hi; ++i)
        for (int64_t j = 0; j < jb->N; ++j) {
            double s = dot_f64(jb->A, jb->B, i, j, jb->K);
            if (jb->S)
                jb->S[i * jb->N + j] = s;
            if (jb->C) {
                uint16_t *c = &jb->C[i * jb->N + j];
                if (jb->ep.on)
                    s = apply_epilogue(&jb->ep, s, *c, j);
                *c = oracle_double_to_fp16(s);
            }
        }
    return NULL;
}

/* Runs rows [0, M) split over `nthreads` threads (1 if nthreads < 1). */
static int run_rows(const uint16_t *A, const uint16_t *B, uint16_t *C, double *S,
                    int64_t M, int64_t N, int64_t K, int nthreads, struct epilogue ep)
{
    pthread_once(&g_decode_once, fill_decode_table);
    if (M <= 0 || N <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > M)
        nthreads = (int)M;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    struct rows_job *jobs = (struct rows_job *)calloc((size_t)nthreads, sizeof(struct rows_job));
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return -1;
    }
    char *live = (char *)calloc((size_t)nthreads, 1);
    if (!live) {
        free(th);
        free(jobs);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        struct rows_job jb = {A, B, C, S, M, N, K, M * t / nthreads, M * (t + 1) / nthreads, ep};
        jobs[t] = jb;
        if (t == 0)
            continue;
        if (pthread_create(&th[t], NULL, rows_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            rows_worker(&jobs[t]);   /* could not start a thread: do it here */
    }
    rows_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (live[t])
            pthread_join(th[t], NULL);
    free(live);
    free(th);
    free(jobs);
    return 0;
}

/* C (M×N row-major FP16) = A·B as defined above. Returns 0, or -1 if memory
 * for the thread bookkeeping could not be had. */
int oracle_hgemm(const uint16_t *A, const uint16_t *B, uint16_t *C,
                 int64_t M, int64_t N, int64_t K, int nthreads)
{
    const struct epilogue none = {0, 1.0, 0.0, NULL, 0};
    return run_rows(A, B, C, NULL, M, N, K, nthreads, none);
}

/* The fused variant defined above: C is read (when beta != 0) and
 * overwritten in place. */
int oracle_hgemm_ex(const uint16_t *A, const uint16_t *B, uint16_t *C,
                    int64_t M, int64_t N, int64_t K, double alpha, double beta,
                    const uint16_t *bias, int relu, int nthreads)
{
    const struct epilogue ep = {1, alpha, beta, bias, relu};
    return run_rows(A, B, C, NULL, M, N, K, nthreads, ep);
}

/* The FP64 sums before the final rounding (M×N row-major doubles). */
int oracle_hgemm_sums_f64(const uint16_t *A, const uint16_t *B, double *S,
                          int64_t M, int64_t N, int64_t K, int nthreads)
{
    const struct epilogue none = {0, 1.0, 0.0, NULL, 0};
    return run_rows(A, B, NULL, S, M, N, K, nthreads, none);
}

/* Selected entries (rows[t], cols[t]) for t < count, for spot checks of
 * shapes too large to compute whole. */
void oracle_hgemm_entries(const uint16_t *A, const uint16_t *B, int64_t K,
                          const int64_t *rows, const int64_t *cols, int64_t count,
                          uint16_t *out)
{
    pthread_once(&g_decode_once, fill_decode_table);
    for (int64_t t = 0; t < count; ++t)
        out[t] = oracle_double_to_fp16(dot_f64(A, B, rows[t], cols[t], K));
}

/* Selected entries of the fused variant: c_old[t] is the previous value of
 * entry (rows[t], cols[t]) (ignored when beta == 0; may then be NULL), bias
 * has length N or is NULL. */
void oracle_hgemm_entries_ex(const uint16_t *A, const uint16_t *B, int64_t K,
                             const int64_t *rows, const int64_t *cols, int64_t count,
                             double alpha, double beta, const uint16_t *c_old,
                             const uint16_t *bias, int relu, uint16_t *out)
{
    pthread_once(&g_decode_once, fill_decode_table);
    const struct epilogue ep = {1, alpha, beta, bias, relu};
    for (int64_t t = 0; t < count; ++t) {
        const double s = dot_f64(A, B, rows[t], cols[t], K);
        out[t] = oracle_double_to_fp16(apply_epilogue(&ep, s, c_old ? c_old[t] : 0, cols[t]));
    }
}

/* ---- the triangular product ---------------------------------------------
 *
 * "异构计算中高性能TRMM与TRSM的递归算法实现", §2.2: left side, lower triangle,
 * transposed (B ← alpha·Aᵀ·B), computed out of place, every matrix
 * column-major as on the page:
 *
 *     C(i,j) = fp16_rne( alpha · Σ_{k=i}^{n-1} A(k,i) · B(k,j) )
 *
 * with A(r,c) = A[c*lda + r], B(r,j) = B[j*ldb + r], C(r,j) = C[j*ldc + r].
 * Only the lower triangle of A (row k ≥ column i) is read. The sum runs in
 * increasing k in FP64 and is rounded once: the plain definition, not the
 * page's recursion (which reaches the same value up to rounding). */

struct trmm_job {
    const uint16_t *A, *B;
    uint16_t *C;
    int64_t lda, ldb, ldc, n;
    double alpha;
    int64_t col_lo, col_hi;
};

static void *trmm_worker(void *arg)
{
    const struct trmm_job *jb = (const struct trmm_job *)arg;
    for (int64_t j = jb->col_lo; j < jb->col_hi; ++j)
        for (int64_t i = 0; i < jb->n; ++i) {
            double s = 0.0;
            for (int64_t k = i; k < jb->n; ++k)
                s += g_decode[jb->A[i * jb->lda + k]] * g_decode[jb->B[j * jb->ldb + k]];
            jb->C[j * jb->ldc + i] = oracle_double_to_fp16(jb->alpha * s);
        }
    return NULL;
}

int oracle_trmm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, uint16_t *C,
                int64_t ldc, int64_t n, int64_t m, double alpha, int nthreads)
{
    pthread_once(&g_decode_once, fill_decode_table);
    if (n <= 0 || m <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > m)
        nthreads = (int)m;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    struct trmm_job *jobs = (struct trmm_job *)calloc((size_t)nthreads, sizeof(struct trmm_job));
    char *live = (char *)calloc((size_t)nthreads, 1);
    if (!th || !jobs || !live) {
        free(th);
        free(jobs);
        free(live);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        struct trmm_job jb = {A, B, C, lda, ldb, ldc, n, alpha, m * t / nthreads, m * (t + 1) / nthreads};
        jobs[t] = jb;
        if (t == 0)
            continue;
        if (pthread_create(&th[t], NULL, trmm_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            trmm_worker(&jobs[t]);
    }
    trmm_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (live[t])
            pthread_join(th[t], NULL);
    free(live);
    free(th);
    free(jobs);
    return 0;
}

/* ---- the triangular solve ------------------------------------------------
 *
 * "异构计算中高性能TRMM与TRSM的递归算法实现", §2.3 (TRSM: solve for X), in the
 * same variant as the triangular product above (left side, lower triangle,
 * transposed), out of place, every matrix column-major:
 *
 *     Aᵀ · X = alpha · B,   X(i,j) = fp16_rne( x_i )  for each column j
 *
 * where x solves the upper-triangular system Aᵀ x = alpha·b in FP64 by back
 * substitution, x_i = (alpha·b_i − Σ_{k>i} A(k,i)·x_k) / A(i,i), k in
 * increasing order, rounded once at the end. Only the lower triangle of A
 * (row ≥ column) is read; a zero on the diagonal gives ±Inf or NaN, as the
 * division does. */

struct trsm_job {
    const uint16_t *A, *B;
    uint16_t *X;
    int64_t lda, ldb, ldx, n;
    double alpha;
    int64_t col_lo, col_hi;
    double *work;    /* n doubles per job */
    int trans;       /* 1: Aᵀ·X = alpha·B (back substitution); 0: A·X = alpha·B (forward) */
};

static void *trsm_worker(void *arg)
{
    const struct trsm_job *jb = (const struct trsm_job *)arg;
    const int64_t n = jb->n;
    double *x = jb->work;
    for (int64_t j = jb->col_lo; j < jb->col_hi; ++j) {
        if (jb->trans) {
            /* row i of Aᵀ holds A(k,i) for k >= i: last row first */
            for (int64_t i = n - 1; i >= 0; --i) {
                double s = jb->alpha * g_decode[jb->B[j * jb->ldb + i]];
                for (int64_t k = i + 1; k < n; ++k)
                    s -= g_decode[jb->A[i * jb->lda + k]] * x[k];
                x[i] = s / g_decode[jb->A[i * jb->lda + i]];
            }
        } else {
            /* row i of A holds A(i,k) for k <= i: first row first */
            for (int64_t i = 0; i < n; ++i) {
                double s = jb->alpha * g_decode[jb->B[j * jb->ldb + i]];
                for (int64_t k = 0; k < i; ++k)
                    s -= g_decode[jb->A[k * jb->lda + i]] * x[k];
                x[i] = s / g_decode[jb->A[i * jb->lda + i]];
            }
        }
        for (int64_t i = 0; i < n; ++i)
            jb->X[j * jb->ldx + i] = oracle_double_to_fp16(x[i]);
    }
    return NULL;
}

static int trsm_run(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, uint16_t *X,
                    int64_t ldx, int64_t n, int64_t m, double alpha, int nthreads, int trans);

int oracle_trsm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, uint16_t *X,
                int64_t ldx, int64_t n, int64_t m, double alpha, int nthreads)
{
    return trsm_run(A, lda, B, ldb, X, ldx, n, m, alpha, nthreads, 1);
}

/* The page's literal orientation of the solve (§2.3: X = A\B column by
 * column): A·X = alpha·B with the same lower triangle A, untransposed, so
 * row i of the system is sum_{k <= i} A(i,k)·x_k = alpha·b_i, solved by
 * forward substitution, x_i = (alpha·b_i − Σ_{k<i} A(i,k)·x_k) / A(i,i), k
 * increasing, in FP64, each x_i rounded once at the end. Same operands,
 * layout and reading of the lower triangle only as oracle_trsm. */
int oracle_trsm_n(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, uint16_t *X,
                  int64_t ldx, int64_t n, int64_t m, double alpha, int nthreads)
{
    return trsm_run(A, lda, B, ldb, X, ldx, n, m, alpha, nthreads, 0);
}

static int trsm_run(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, uint16_t *X,
                    int64_t ldx, int64_t n, int64_t m, double alpha, int nthreads, int trans)
{
    pthread_once(&g_decode_once, fill_decode_table);
    if (n <= 0 || m <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > m)
        nthreads = (int)m;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    struct trsm_job *jobs = (struct trsm_job *)calloc((size_t)nthreads, sizeof(struct trsm_job));
    char *live = (char *)calloc((size_t)nthreads, 1);
    double *work = (double *)malloc((size_t)nthreads * (size_t)n * sizeof(double));
    if (!th || !jobs || !live || !work) {
        free(th);
        free(jobs);
        free(live);
        free(work);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        struct trsm_job jb = {A, B, X, lda, ldb, ldx, n, alpha, m * t / nthreads, m * (t + 1) / nthreads,
                              work + (size_t)t * (size_t)n, trans};
        jobs[t] = jb;
        if (t == 0)
            continue;
        if (pthread_create(&th[t], NULL, trsm_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            trsm_worker(&jobs[t]);
    }
    trsm_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (live[t])
            pthread_join(th[t], NULL);
    free(work);
    free(live);
    free(th);
    free(jobs);
    return 0;
}
