"""Pins for the oracle, each against something other than the oracle itself.

CPU only. The pins are chosen so that a plausible slip anywhere in the
oracle fails at least one of them: a wrong rounding mode (tie fixtures,
exhaustive codec, numpy rounding), a transposed or mis-indexed operand
(identity operands, non-symmetric brute force), a dropped term (brute force,
integer exactness), FP16-width accumulation (the wide-accumulation fixture),
an overflow or subnormal slip (fixtures, exhaustive codec).
"""

import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle

# ---------------------------------------------------------------------------
# A textbook binary16 rounding on exact rationals, written independently of
# the oracle's frexp/rint code: used by the brute-force pin.


def fraction_to_fp16_bits(x: Fraction) -> int:
    """Round-to-nearest-even of an exact rational to IEEE binary16 bits."""
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a == 0:
        return sign
    # exponent e with 2^e <= a < 2^(e+1), clamped to the subnormal floor -14
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)
    quantum = Fraction(2) ** (e - 10)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    # fl is the significand on the 2^(e-10) grid, in [0, 2048]
    if fl == 2048:
        fl, e = 1024, e + 1
    if e > 15:
        return sign | 0x7C00
    if fl < 1024:  # subnormal (only reachable with e == -14)
        return sign | fl
    return sign | ((e + 15) << 10) | (fl - 1024)


def bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float16).view(np.uint16)


def random_fp16(rng, shape, lo_exp=-6, hi_exp=4):
    """Random FP16 values over several binades, both signs, some zeros."""
    mant = rng.integers(0, 1024, size=shape)
    expo = rng.integers(lo_exp + 15, hi_exp + 15, size=shape)
    sgn = rng.integers(0, 2, size=shape)
    b = (sgn << 15) | (expo << 10) | mant
    b = np.where(rng.random(shape) < 0.05, 0, b)
    return b.astype(np.uint16).view(np.float16)


# ---------------------------------------------------------------------------
# golden fixtures (hand-derived; citations in the file)


def load_golden(path):
    cases, cur = [], None
    with open(path, encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *rest = line.split()
            if tag == "case":
                cur = {"name": rest[0]}
                cases.append(cur)
            elif tag == "dims":
                cur["dims"] = tuple(int(v) for v in rest)
            elif tag in ("A", "B"):
                cur[tag] = [float(v) for v in rest]
            elif tag == "C":
                cur["C"] = [int(v, 16) for v in rest]
    return cases


def test_golden_hand_worked_cases(golden_dir):
    cases = load_golden(os.path.join(golden_dir, "hand_worked_cases.txt"))
    assert len(cases) >= 6
    for cs in cases:
        M, N, K = cs["dims"]
        a = np.array(cs["A"], dtype=np.float64).reshape(M, K)
        b = np.array(cs["B"], dtype=np.float64).reshape(N, K)
        # every fixture value must be exactly representable
        assert np.array_equal(a.astype(np.float16).astype(np.float64), a), cs["name"]
        assert np.array_equal(b.astype(np.float16).astype(np.float64), b), cs["name"]
        c = oracle.hgemm(a.astype(np.float16), b.astype(np.float16))
        got = bits(c).reshape(-1).tolist()
        assert got == cs["C"], (cs["name"], [hex(v) for v in got])


# ---------------------------------------------------------------------------
# the FP16 codec


def test_decode_exhaustive_against_numpy():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(h)) for h in allbits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_encode_roundtrip_exhaustive():
    for h in range(65536):
        e, f = (h >> 10) & 0x1F, h & 0x3FF
        if e == 31 and f:
            continue  # NaN payloads are not preserved
        assert oracle.double_to_fp16(oracle.fp16_to_double(h)) == h, hex(h)


def test_encode_against_numpy_including_exact_midpoints():
    rng = np.random.default_rng(7)
    xs = []
    # every midpoint between adjacent finite FP16 values (exact in float64),
    # and points just either side of it
    pos = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    xs += list(mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, np.inf))
    xs += [65504.0, 65519.99, 65520.0, 65536.0, 1e6, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26]
    xs += list(rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000))
    xs = np.array(xs, dtype=np.float64)
    xs = np.concatenate([xs, -xs])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_fp16(x) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


# ---------------------------------------------------------------------------
# the contraction


def test_bruteforce_exact_rationals_tiny_shapes():
    """With K <= 6 the FP64 sum of FP16 products is exact; the oracle must
    equal the exact rational sum rounded to FP16 (ties to even), bit for bit."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        M, N, K = (int(v) for v in rng.integers(1, 7, size=3))
        a = random_fp16(rng, (M, K))
        b = random_fp16(rng, (N, K))
        got = bits(oracle.hgemm(a, b))
        for i in range(M):
            for j in range(N):
                s = sum(Fraction(float(a[i, k])) * Fraction(float(b[j, k])) for k in range(K))
                assert got[i, j] == fraction_to_fp16_bits(s), (trial, i, j, s)


def test_bruteforce_handmade_ties():
    """Sums built to land exactly on FP16 midpoints at several binades."""
    rnd = random.Random(5)
    for _ in range(200):
        e = rnd.randint(-10, 13)
        q = Fraction(2) ** (e - 10)  # FP16 spacing in binade 2^e
        n = rnd.randint(1024, 2047)
        target = (n + Fraction(1, 2)) * q  # a midpoint
        x = float(n * q)
        y = float(q / 2)
        a = np.array([[x, y]], dtype=np.float16)
        b = np.array([[1.0, 1.0]], dtype=np.float16)
        if float(a[0, 0]) != x or float(a[0, 1]) != y:
            continue  # y underflowed FP16; skip
        got = int(bits(oracle.hgemm(a, b))[0, 0])
        assert got == fraction_to_fp16_bits(target), (e, n)


def test_identity_and_zero_operands():
    rng = np.random.default_rng(3)
    M, K, N = 37, 29, 23
    b = random_fp16(rng, (N, K))
    # A = I (M = K): C[i, j] = B[i, j] = b[j, i]
    eye_k = np.eye(K, dtype=np.float16)
    c = oracle.hgemm(eye_k, b)
    assert np.array_equal(bits(c), bits(b.T))
    # B = I (K = N): C = A exactly
    a = random_fp16(rng, (M, K))
    c = oracle.hgemm(a, np.eye(K, dtype=np.float16))
    assert np.array_equal(bits(c), bits(a))
    # zeros give +0 everywhere
    assert np.all(bits(oracle.hgemm(np.zeros((M, K), np.float16), b)) == 0)
    assert np.all(bits(oracle.hgemm(a, np.zeros((N, K), np.float16))) == 0)
    # a permutation picks single columns, in order
    perm = rng.permutation(K)
    p = np.zeros((K, K), dtype=np.float16)
    p[np.arange(K), perm] = 1
    c = oracle.hgemm(p, b)  # C[i, j] = b[j, perm[i]]
    assert np.array_equal(bits(c), bits(b[:, perm].T))


def test_rank_one_closed_form():
    """A = 1 (all ones), column j of B constant c_j: C[i, j] = K * c_j."""
    M, N, K = 5, 7, 12
    cvals = np.array([0.5, -1.25, 3.0, 0.0, 2.0, -0.75, 8.0], dtype=np.float16)
    a = np.ones((M, K), dtype=np.float16)
    b = np.repeat(cvals[:, None], K, axis=1)
    c = oracle.hgemm(a, b).astype(np.float64)
    assert np.array_equal(c, np.tile(K * cvals.astype(np.float64), (M, 1)))


@pytest.mark.parametrize("M,N,K", [(17, 13, 256), (64, 64, 256), (100, 3, 250)])
def test_integer_operands_equal_int64_product(M, N, K):
    """Entries in {-2..2} with K <= 256: |C| <= 1024, every value exact."""
    rng = np.random.default_rng(M * 1000 + N)
    ai = rng.integers(-2, 3, size=(M, K))
    bi = rng.integers(-2, 3, size=(N, K))
    c = oracle.hgemm(ai.astype(np.float16), bi.astype(np.float16))
    assert np.array_equal(c.astype(np.int64), ai @ bi.T)


@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (256, 8, 1000)])
def test_fp64_sums_against_numpy_matmul(M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = (2 * rng.random((M, K)) - 1).astype(np.float16)
    b = (2 * rng.random((N, K)) - 1).astype(np.float16)
    s = oracle.sums_f64(a, b)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    scale = np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64)).T
    assert np.all(np.abs(s - ref) <= 1e-12 * np.maximum(scale, 1e-300))
    # the FP16 result is the sums rounded, element by element
    c = oracle.hgemm(a, b)
    assert np.array_equal(bits(c), bits(s.astype(np.float16)))


def test_entries_and_threads_agree_with_full_product():
    rng = np.random.default_rng(17)
    a = (2 * rng.random((45, 130)) - 1).astype(np.float16)
    b = (2 * rng.random((33, 130)) - 1).astype(np.float16)
    full = oracle.hgemm(a, b, nthreads=1)
    for nt in (2, 5, 64):
        assert np.array_equal(bits(oracle.hgemm(a, b, nthreads=nt)), bits(full))
    rows = rng.integers(0, 45, size=200)
    cols = rng.integers(0, 33, size=200)
    assert np.array_equal(bits(oracle.entries(a, b, rows, cols)), bits(full[rows, cols]))


def test_degenerate_shapes():
    a = np.zeros((0, 5), np.float16)
    b = np.ones((4, 5), np.float16)
    assert oracle.hgemm(a, b).shape == (0, 4)
    # K = 0: every entry is the empty sum, +0
    c = oracle.hgemm(np.zeros((3, 0), np.float16), np.zeros((2, 0), np.float16))
    assert c.shape == (3, 2) and np.all(bits(c) == 0)
    with pytest.raises(ValueError):
        oracle.hgemm(np.zeros((3, 4), np.float16), np.zeros((2, 5), np.float16))


# ---------------------------------------------------------------------------
# the fused variant: fp16(f(alpha·A·B + beta·C_old + bias[j])), f = ReLU or id


def test_fused_reduces_to_the_plain_product():
    """alpha = 1, beta = 0, no bias, no ReLU is the plain product, bit for bit."""
    rng = np.random.default_rng(31)
    a = random_fp16(rng, (37, 53))
    b = random_fp16(rng, (29, 53))
    assert np.array_equal(bits(oracle.hgemm_ex(a, b)), bits(oracle.hgemm(a, b)))


@pytest.mark.parametrize("alpha,beta,relu", [(1.0, 1.0, False), (2.0, -1.0, True), (-0.5, 2.0, False),
                                             (1.0, 0.0, True), (0.5, 0.5, True), (-1.0, 0.0, False)])
def test_fused_integer_operands_exact(alpha, beta, relu):
    """Integer A, B, C_old and bias with power-of-two alpha and beta: every
    value is an exact multiple of 1/4 well inside FP16's integer range, so the
    oracle must equal exact rational arithmetic on an int64 product; M != N
    and a bias that differs per column catch a bias indexed by row or a
    transposed C."""
    rng = np.random.default_rng(int(100 * alpha + 10 * beta + relu) & 0xFFFF)
    M, N, K = 23, 17, 48
    ai = rng.integers(-2, 3, size=(M, K))
    bi = rng.integers(-2, 3, size=(N, K))
    ci = rng.integers(-60, 61, size=(M, N))
    bias = rng.integers(-20, 21, size=N)
    prod = ai.astype(np.int64) @ bi.astype(np.int64).T
    want = np.empty((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            v = Fraction(alpha) * int(prod[i, j]) + Fraction(beta) * int(ci[i, j]) + int(bias[j])
            if relu and v < 0:
                v = Fraction(0)
            want[i, j] = fraction_to_fp16_bits(v)
    got = oracle.hgemm_ex(ai.astype(np.float16), bi.astype(np.float16), ci.astype(np.float16),
                          alpha=alpha, beta=beta, bias=bias.astype(np.float16), relu=relu)
    g = bits(got)
    zero = (want & 0x7FFF) == 0
    assert np.array_equal(g[~zero], want[~zero])
    assert np.all((g[zero] & 0x7FFF) == 0)


def test_fused_rounds_once():
    """S = 1024·2 + 1·1 = 2049 and C_old = 1: the exact 2050 is an FP16 value;
    rounding S first (2049 -> 2048) and then adding would give 2049 -> 2048."""
    a = np.array([[1024.0, 1.0]], np.float16)
    b = np.array([[2.0, 1.0]], np.float16)
    c = np.array([[1.0]], np.float16)
    got = oracle.hgemm_ex(a, b, c, beta=1.0)
    assert float(got[0, 0]) == 2050.0
    assert float(oracle.hgemm(a, b)[0, 0]) == 2048.0   # 2049 alone is a tie to even


def test_fused_beta_zero_does_not_read_c():
    rng = np.random.default_rng(5)
    a = random_fp16(rng, (9, 16))
    b = random_fp16(rng, (7, 16))
    bias = random_fp16(rng, (7,))
    nan_c = np.full((9, 7), np.nan, np.float16)
    got = oracle.hgemm_ex(a, b, nan_c, alpha=1.5, beta=0.0, bias=bias, relu=True)
    assert not np.isnan(got.astype(np.float32)).any()
    assert np.array_equal(bits(got), bits(oracle.hgemm_ex(a, b, None, alpha=1.5, bias=bias, relu=True)))
    assert np.all(got.astype(np.float32) >= 0)


def test_fused_entries_agree_with_full_product():
    rng = np.random.default_rng(77)
    a = random_fp16(rng, (40, 96))
    b = random_fp16(rng, (33, 96))
    c = random_fp16(rng, (40, 33))
    bias = random_fp16(rng, (33,))
    full = oracle.hgemm_ex(a, b, c, alpha=0.75, beta=-1.25, bias=bias, relu=True, nthreads=3)
    rows = rng.integers(0, 40, 200)
    cols = rng.integers(0, 33, 200)
    part = oracle.entries_ex(a, b, rows, cols, c, alpha=0.75, beta=-1.25, bias=bias, relu=True)
    assert np.array_equal(bits(part), bits(full[rows, cols]))


# ---------------------------------------------------------------------------
# the triangular product of the TRMM page: C = fp16(alpha·Aᵀ·B), A lower


def test_trmm_bruteforce_exact_rationals():
    rng = np.random.default_rng(41)
    for n, m in [(1, 1), (2, 3), (3, 2), (5, 4), (6, 6)]:
        a = random_fp16(rng, (n, n))
        b = random_fp16(rng, (n, m))
        got = bits(oracle.trmm(a, b, alpha=0.75))
        for i in range(n):
            for j in range(m):
                v = Fraction(0)
                for k in range(i, n):    # A(k, i) with k >= i: the lower triangle
                    v += Fraction(float(a[k, i])) * Fraction(float(b[k, j]))
                assert got[i, j] == fraction_to_fp16_bits(Fraction(0.75) * v), (n, m, i, j)


def test_trmm_against_numpy_and_plain_product():
    rng = np.random.default_rng(42)
    n, m = 70, 33
    a = rng.uniform(0, 1, size=(n, n)).astype(np.float16)
    b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
    got = oracle.trmm(a, b)
    ref = np.tril(a.astype(np.float64)).T @ b.astype(np.float64)
    assert np.allclose(got.astype(np.float64), ref, rtol=2.0 ** -10, atol=0)
    # with zeros above the diagonal the plain product (already pinned) is the same:
    # Cᵀ = Bᵀ·A, i.e. hgemm(a_op = Bᵀ, b_op rows = columns of A)
    lower = np.tril(a)
    plain = oracle.hgemm(np.ascontiguousarray(b.T), np.ascontiguousarray(lower.T)).T
    assert np.array_equal(bits(got), bits(plain))


def test_trmm_reads_only_the_lower_triangle():
    rng = np.random.default_rng(43)
    n, m = 40, 9
    a = rng.uniform(-1, 1, size=(n, n)).astype(np.float16)
    b = rng.uniform(-1, 1, size=(n, m)).astype(np.float16)
    poisoned = a.copy()
    poisoned[np.triu_indices(n, 1)] = np.nan
    assert np.array_equal(bits(oracle.trmm(poisoned, b)), bits(oracle.trmm(a, b)))


def test_trmm_identity_and_scaling():
    rng = np.random.default_rng(44)
    n, m = 17, 5
    b = random_fp16(rng, (n, m))
    eye = np.eye(n, dtype=np.float16)
    assert np.array_equal(bits(oracle.trmm(eye, b)), bits(b))
    assert np.array_equal(bits(oracle.trmm(eye, b, alpha=2.0)), bits((b.astype(np.float64) * 2).astype(np.float16)))


# ---------------------------------------------------------------------------
# the triangular solve: Aᵀ·X = alpha·B, A lower


def well_conditioned_lower(rng, n):
    """Diagonal in [1, 2), strictly lower part in [0, 1/n): a diagonally
    dominant triangle, so the solve is well conditioned."""
    a = (rng.uniform(0, 1, size=(n, n)) / n).astype(np.float16)
    a[np.diag_indices(n)] = rng.uniform(1, 2, size=n).astype(np.float16)
    return a


def test_trsm_against_scipy_and_residual():
    import scipy.linalg
    rng = np.random.default_rng(51)
    n, m = 90, 21
    a = well_conditioned_lower(rng, n)
    b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
    x = oracle.trsm(a, b, alpha=1.5)
    lower = np.tril(a.astype(np.float64))
    ref = scipy.linalg.solve_triangular(lower.T, 1.5 * b.astype(np.float64), lower=False)
    # one rounding of the exact FP64 solution
    assert np.array_equal(bits(x), bits(ref.astype(np.float16)))
    # the rounded solution satisfies the system up to FP16 rounding
    resid = lower.T @ x.astype(np.float64) - 1.5 * b.astype(np.float64)
    assert np.max(np.abs(resid)) < 4 * 2.0 ** -11 * np.max(np.abs(1.5 * b.astype(np.float64))) + 1e-3


def test_trsm_bruteforce_exact_rationals():
    rng = np.random.default_rng(52)
    for n, m in [(1, 1), (2, 2), (4, 3), (6, 2)]:
        a = well_conditioned_lower(rng, n)
        b = random_fp16(rng, (n, m))
        got = bits(oracle.trsm(a, b, alpha=0.5))
        for j in range(m):
            x = [Fraction(0)] * n
            for i in range(n - 1, -1, -1):
                s = Fraction(0.5) * Fraction(float(b[i, j]))
                for k in range(i + 1, n):
                    s -= Fraction(float(a[k, i])) * x[k]
                x[i] = s / Fraction(float(a[i, i]))
            for i in range(n):
                assert got[i, j] == fraction_to_fp16_bits(x[i]), (n, m, i, j)


def test_trsm_inverts_trmm_and_ignores_the_upper_triangle():
    rng = np.random.default_rng(53)
    n, m = 48, 7
    a = well_conditioned_lower(rng, n)
    eye = np.eye(n, dtype=np.float16)
    b = random_fp16(rng, (n, m))
    assert np.array_equal(bits(oracle.trsm(eye, b, alpha=2.0)),
                          bits((b.astype(np.float64) * 2).astype(np.float16)))
    poisoned = a.copy()
    poisoned[np.triu_indices(n, 1)] = np.nan
    assert np.array_equal(bits(oracle.trsm(poisoned, b)), bits(oracle.trsm(a, b)))
    # solving against the product recovers the right-hand side (to FP16 rounding)
    c = oracle.trmm(a, b)
    back = oracle.trsm(a, c).astype(np.float64)
    assert np.allclose(back, b.astype(np.float64), rtol=1e-2, atol=1e-2)


# ---- the solve in the page's literal orientation, A·X = alpha·B (forward substitution)

def test_trsm_n_against_scipy_and_residual():
    import scipy.linalg
    rng = np.random.default_rng(61)
    n, m = 90, 21
    a = well_conditioned_lower(rng, n)
    b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
    x = oracle.trsm_n(a, b, alpha=1.5)
    lower = np.tril(a.astype(np.float64))
    ref = scipy.linalg.solve_triangular(lower, 1.5 * b.astype(np.float64), lower=True)
    # one rounding of the exact FP64 solution
    assert np.array_equal(bits(x), bits(ref.astype(np.float16)))
    resid = lower @ x.astype(np.float64) - 1.5 * b.astype(np.float64)
    assert np.max(np.abs(resid)) < 4 * 2.0 ** -11 * np.max(np.abs(1.5 * b.astype(np.float64))) + 1e-3
    # not the transposed system: a wrong orientation fails the residual
    wrong = oracle.trsm(a, b, alpha=1.5).astype(np.float64)
    assert np.max(np.abs(lower @ wrong - 1.5 * b.astype(np.float64))) > 1e-2


def test_trsm_n_bruteforce_exact_rationals():
    rng = np.random.default_rng(62)
    for n, m in [(1, 1), (2, 2), (4, 3), (6, 2)]:
        a = well_conditioned_lower(rng, n)
        b = random_fp16(rng, (n, m))
        got = bits(oracle.trsm_n(a, b, alpha=0.5))
        for j in range(m):
            x = [Fraction(0)] * n
            for i in range(n):
                s = Fraction(0.5) * Fraction(float(b[i, j]))
                for k in range(i):
                    s -= Fraction(float(a[i, k])) * x[k]
                x[i] = s / Fraction(float(a[i, i]))
            for i in range(n):
                assert got[i, j] == fraction_to_fp16_bits(x[i]), (n, m, i, j)


def test_trsm_n_special_cases_and_the_reversed_transposed_system():
    rng = np.random.default_rng(63)
    n, m = 48, 7
    a = well_conditioned_lower(rng, n)
    eye = np.eye(n, dtype=np.float16)
    b = random_fp16(rng, (n, m))
    assert np.array_equal(bits(oracle.trsm_n(eye, b, alpha=2.0)),
                          bits((b.astype(np.float64) * 2).astype(np.float16)))
    poisoned = a.copy()
    poisoned[np.triu_indices(n, 1)] = np.nan
    assert np.array_equal(bits(oracle.trsm_n(poisoned, b)), bits(oracle.trsm_n(a, b)))
    # With J the order reversal, A·X = B is (J·Aᵀ·J)ᵀ·(J·X) = J·B, the
    # transposed system of the lower triangle J·Aᵀ·J: the already-pinned
    # transposed solve gives the same solution up to the summation order
    # (within one FP16 step of each other).
    rev = np.ascontiguousarray(a.T[::-1, ::-1])
    other = oracle.trsm(rev, np.ascontiguousarray(b[::-1]))[::-1].astype(np.float64)
    mine = oracle.trsm_n(a, b).astype(np.float64)
    assert np.all(np.abs(mine - other) <= 2.0 ** -10 * np.maximum(np.abs(mine), 2.0 ** -14))
