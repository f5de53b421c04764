"""Seeded synthetic operands for the FP16 HGEMM C = A·B.

This module is shared by the tests and the benchmark. It holds no arithmetic
of the method itself (no products, no sums, no output rounding): it only
draws the two operands, so that the oracle and the CUDA path can be fed the
same bytes.

Layouts follow the problem statement of "Nvidia Tensor Core-MMA PTX编程入门",
§4 示例: A is M×K row-major (element (i, k) at A[i*K + k]) and B is K×N
column-major, stored as N columns of K contiguous values (element (k, j) at
B[j*K + k]). Both arrays are returned as ``numpy.float16`` in that storage
order.

Random numbers come from splitmix64 in counter form: draw number t of a
stream with seed s is mix(s + (t + 1)·γ) with γ = 0x9E3779B97F4A7C15 and mix
the splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014). A uniform in [0, 1) is the top
53 bits scaled by 2^-53. The A stream uses draws 0 .. M*K-1 in A's storage
order; the B stream continues with draws M*K .. M*K+N*K-1 in B's storage
order (Gaussian draws take two uniforms per value, so their counters double).

Value recipes (the workloads of the benchmark configurations):
  * ``uniform``  : 2u - 1 rounded to the nearest FP16 (ties to even);
  * ``int``      : floor(5u) - 2, i.e. integers uniform in {-2, ..., 2};
  * ``normal``   : Box-Muller on consecutive uniform pairs
                   z = sqrt(-2 ln(1 - u1)) * cos(2π u2); A ~ N(0, 1) and
                   B ~ N(0, 1)/sqrt(K), each rounded to FP16;
  * ``normal_both``: the same draws with both operands scaled by 1/sqrt(K)
                   (the literal reading of "N(0,1) values scaled by
                   1/sqrt(K)"; C then has standard deviation 1/sqrt(K));
  * ``unit``     : u rounded to the nearest FP16 (values in [0, 1]), like
                   the rand(Float32) operands of the TRMM page's example (§5.1).

The triangular product (``trmm_operands``) takes A (n×n, its lower triangle
is the operand) and B (n×m), both column-major as on the TRMM page: arrays of
n columns (A) and m columns (B) of n contiguous values. A's stream uses draws
0 .. n*n-1, B's continues after it.

The triangular solve (``trsm_operands``) needs a triangle that is well
conditioned in FP16, which a uniform [0, 1) triangle is not (its inverse
grows exponentially with n). Its A takes the same draws u, as 1 + u on the
diagonal and u / n elsewhere (a diagonally dominant triangle: every column
of the strict lower part sums to less than 1 ≤ the diagonal); B is ``unit``.
"""

from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# chunking keeps the float64 temporaries of the 8192 x 8192 operands bounded
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the splitmix64 stream ``seed``."""
    t = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + t * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """u = (x >> 11) · 2^-53, exactly representable in float64, in [0, 1)."""
    x = splitmix64(seed, start, count)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _fill(seed: int, start: int, count: int, kind: str, scale: float) -> np.ndarray:
    out = np.empty(count, dtype=np.float16)
    per = 2 if kind in ("normal", "normal_both") else 1
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        if kind == "uniform":
            v = 2.0 * uniform01(seed, start + lo, n) - 1.0
        elif kind == "unit":
            v = uniform01(seed, start + lo, n)
        elif kind == "int":
            v = np.floor(5.0 * uniform01(seed, start + lo, n)) - 2.0
        elif kind in ("normal", "normal_both"):
            u = uniform01(seed, start + per * lo, per * n)
            u1, u2 = u[0::2], u[1::2]
            v = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2) * scale
        else:
            raise ValueError(f"unknown value kind {kind!r}")
        out[lo:lo + n] = v.astype(np.float16)
    return out


def operands(M: int, N: int, K: int, seed: int, kind: str = "uniform"):
    """Returns (A, B): A as an (M, K) array, B as an (N, K) array whose row j
    is column j of the K×N operand, both float16 and C-contiguous."""
    per = 2 if kind in ("normal", "normal_both") else 1
    b_scale = 1.0 / np.sqrt(K) if (kind in ("normal", "normal_both") and K > 0) else 1.0
    a_scale = 1.0 / np.sqrt(K) if (kind == "normal_both" and K > 0) else 1.0
    a = _fill(seed, 0, M * K, kind, a_scale).reshape(M, K)
    b = _fill(seed, per * M * K, N * K, kind, b_scale).reshape(N, K)
    return a, b


# The benchmark workloads, each named by what it is. The integer variant of
# the 256-cube uses the same shape with the seed offset by 100.
WORKLOADS = {
    "hgemm_256": dict(M=256, N=256, K=256, kind="uniform", seed=1000),
    "hgemm_256_int": dict(M=256, N=256, K=256, kind="int", seed=1100),
    "hgemm_2048": dict(M=2048, N=2048, K=2048, kind="uniform", seed=1001),
    "hgemm_1000_ragged": dict(M=1000, N=1000, K=1000, kind="uniform", seed=1002),
    "hgemm_8192": dict(M=8192, N=8192, K=8192, kind="normal", seed=1003),
    # the same draws with A scaled as well (a secondary parity case)
    "hgemm_8192_both_scaled": dict(M=8192, N=8192, K=8192, kind="normal_both", seed=1003),
    "hgemm_4096x256x4096_skinny": dict(M=4096, N=256, K=4096, kind="uniform", seed=1004),
    # the TRMM page's shapes: 8192×8192 (its measurements, §4.2) and A 4096×4096
    # with a 4096×256 right-hand side (its example, §5.1)
    "trmm_8192": dict(op="trmm", n=8192, m=8192, kind="unit", seed=1005),
    "trmm_4096x256": dict(op="trmm", n=4096, m=256, kind="unit", seed=1006),
    # the solve on the same shapes (§4.2 times it at 8192×8192)
    "trsm_8192": dict(op="trsm", n=8192, m=8192, kind="dominant", seed=1007),
    "trsm_4096x256": dict(op="trsm", n=4096, m=256, kind="dominant", seed=1008),
    # the same operands solved in the page's literal orientation, A·X = B
    "trsm_n_8192": dict(op="trsm_n", n=8192, m=8192, kind="dominant", seed=1007),
    "trsm_n_4096x256": dict(op="trsm_n", n=4096, m=256, kind="dominant", seed=1008),
}


def trmm_operands(n: int, m: int, seed: int, kind: str = "unit"):
    """(a_col, b_col): a_col (n, n) holds column c of A in row c (the whole
    square is drawn; only its lower triangle, row >= column, is the operand),
    b_col (m, n) holds column j of B in row j."""
    a = _fill(seed, 0, n * n, kind, 1.0).reshape(n, n)
    b = _fill(seed, n * n, m * n, kind, 1.0).reshape(m, n)
    return a, b


def trsm_operands(n: int, m: int, seed: int, c: float = 1.0):
    """(a_col, b_col) as for trmm_operands, with the diagonally dominant A
    (c = 1). c > 1 scales the strict lower part to c·u/n: column sums up to
    c, a triangle that is no longer diagonally dominant for c > 1."""
    a = np.empty(n * n, dtype=np.float16)
    for lo in range(0, n * n, _CHUNK):
        cnt = min(_CHUNK, n * n - lo)
        u = uniform01(seed, lo, cnt)
        idx = np.arange(lo, lo + cnt)
        diag = (idx // n) == (idx % n)
        a[lo:lo + cnt] = np.where(diag, 1.0 + u, c * u / n).astype(np.float16)
    b = _fill(seed, n * n, m * n, "unit", 1.0).reshape(m, n)
    return a.reshape(n, n), b


def workload(name: str):
    """(A, B, spec) for a named workload."""
    spec = WORKLOADS[name]
    if spec.get("op") == "trmm":
        a, b = trmm_operands(spec["n"], spec["m"], spec["seed"], spec["kind"])
        return a, b, spec
    if spec.get("op") in ("trsm", "trsm_n"):
        a, b = trsm_operands(spec["n"], spec["m"], spec["seed"])
        return a, b, spec
    a, b = operands(spec["M"], spec["N"], spec["K"], spec["seed"], spec["kind"])
    return a, b, spec
