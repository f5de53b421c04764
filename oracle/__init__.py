"""The oracle for the FP16 HGEMM, C = A·B (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product path in
``tensor_core_dense_fp16_gb300`` never does, and the two share no code.

The arithmetic lives in ``hgemm_oracle.c`` (plain C, FP64 sum in increasing
k, one round-to-nearest-even to FP16 at the end); this module only compiles
it with gcc and marshals numpy arrays into it.

Pins: every function here is pinned in ``tests/test_oracle.py`` against
things other than itself (exact rational arithmetic on tiny shapes, identity
and zero operands, integer operands against an int64 product, numpy's FP64
matmul, numpy's FP16 rounding, and the hand-derived fixtures in
``tests/golden/``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hgemm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-pthread"]

_lib = None


def build(force: bool = False) -> str:
    """Compiles liboracle.so with gcc if it is missing or older than its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, u16p, f64p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        lib.oracle_hgemm.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int]
        lib.oracle_hgemm.restype = ctypes.c_int
        lib.oracle_hgemm_sums_f64.argtypes = [u16p, u16p, f64p, i64, i64, i64, ctypes.c_int]
        lib.oracle_hgemm_sums_f64.restype = ctypes.c_int
        lib.oracle_hgemm_entries.argtypes = [u16p, u16p, i64, ctypes.c_void_p,
                                             ctypes.c_void_p, i64, u16p]
        lib.oracle_hgemm_entries.restype = None
        lib.oracle_hgemm_ex.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_double,
                                        ctypes.c_double, u16p, ctypes.c_int, ctypes.c_int]
        lib.oracle_hgemm_ex.restype = ctypes.c_int
        lib.oracle_hgemm_entries_ex.argtypes = [u16p, u16p, i64, ctypes.c_void_p, ctypes.c_void_p,
                                                i64, ctypes.c_double, ctypes.c_double, u16p, u16p,
                                                ctypes.c_int, u16p]
        lib.oracle_hgemm_entries_ex.restype = None
        lib.oracle_trmm.argtypes = [u16p, i64, u16p, i64, u16p, i64, i64, i64, ctypes.c_double,
                                    ctypes.c_int]
        lib.oracle_trmm.restype = ctypes.c_int
        lib.oracle_trsm.argtypes = [u16p, i64, u16p, i64, u16p, i64, i64, i64, ctypes.c_double,
                                    ctypes.c_int]
        lib.oracle_trsm.restype = ctypes.c_int
        lib.oracle_trsm_n.argtypes = lib.oracle_trsm.argtypes
        lib.oracle_trsm_n.restype = ctypes.c_int
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_fp16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_fp16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def _operands(a, b):
    a = np.ascontiguousarray(a, dtype=np.float16)
    b = np.ascontiguousarray(b, dtype=np.float16)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("a must be (M, K) and b (N, K): row j of b is column j of B")
    return a, b


def hgemm(a: np.ndarray, b: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """C (M, N) float16 for A = a (M, K) and B whose column j is b[j] (b is (N, K))."""
    a, b = _operands(a, b)
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), dtype=np.float16)
    rc = _load().oracle_hgemm(a.ctypes.data, b.ctypes.data, c.ctypes.data, M, N, K,
                              _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_hgemm could not allocate its thread bookkeeping")
    return c


def sums_f64(a: np.ndarray, b: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """The FP64 sums before the final rounding, (M, N) float64."""
    a, b = _operands(a, b)
    M, K = a.shape
    N = b.shape[0]
    s = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_hgemm_sums_f64(a.ctypes.data, b.ctypes.data, s.ctypes.data, M, N, K,
                                       _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_hgemm_sums_f64 could not allocate its thread bookkeeping")
    return s


def entries(a: np.ndarray, b: np.ndarray, rows, cols) -> np.ndarray:
    """C[rows[t], cols[t]] for each t, float16; for shapes too large to do whole."""
    a, b = _operands(a, b)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols must have the same length")
    if rows.size and (rows.min() < 0 or rows.max() >= a.shape[0]
                      or cols.min() < 0 or cols.max() >= b.shape[0]):
        raise IndexError("entry index out of range")
    out = np.empty(rows.shape, dtype=np.float16)
    _load().oracle_hgemm_entries(a.ctypes.data, b.ctypes.data, a.shape[1], rows.ctypes.data,
                                 cols.ctypes.data, rows.size, out.ctypes.data)
    return out


def _epilogue_inputs(c, bias, shape, beta):
    M, N = shape
    if beta != 0.0:
        if c is None:
            raise ValueError("beta != 0 reads C: pass c")
        c = np.ascontiguousarray(c, dtype=np.float16)
        if c.shape != (M, N):
            raise ValueError("c must be (M, N)")
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float16)
        if bias.shape != (N,):
            raise ValueError("bias must have length N")
    return c, bias


def hgemm_ex(a: np.ndarray, b: np.ndarray, c: np.ndarray | None = None, alpha: float = 1.0,
             beta: float = 0.0, bias: np.ndarray | None = None, relu: bool = False,
             nthreads: int | None = None) -> np.ndarray:
    """The fused product, (M, N) float16:
    fp16(f(alpha·A·B + beta·c + bias[j])), f = ReLU if relu; c is not read when beta == 0."""
    a, b = _operands(a, b)
    M, K = a.shape
    N = b.shape[0]
    c, bias = _epilogue_inputs(c, bias, (M, N), beta)
    out = np.array(c, dtype=np.float16, copy=True) if c is not None else np.zeros((M, N), np.float16)
    rc = _load().oracle_hgemm_ex(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K,
                                 float(alpha), float(beta),
                                 bias.ctypes.data if bias is not None else None, int(bool(relu)),
                                 _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_hgemm_ex could not allocate its thread bookkeeping")
    return out


def entries_ex(a: np.ndarray, b: np.ndarray, rows, cols, c: np.ndarray | None = None,
               alpha: float = 1.0, beta: float = 0.0, bias: np.ndarray | None = None,
               relu: bool = False) -> np.ndarray:
    """Entries (rows[t], cols[t]) of the fused product; c is the whole previous C."""
    a, b = _operands(a, b)
    M, K = a.shape
    N = b.shape[0]
    c, bias = _epilogue_inputs(c, bias, (M, N), beta)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols must have the same length")
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise IndexError("entry index out of range")
    c_old = np.ascontiguousarray(c[rows, cols]) if c is not None else None
    out = np.empty(rows.shape, dtype=np.float16)
    _load().oracle_hgemm_entries_ex(a.ctypes.data, b.ctypes.data, K, rows.ctypes.data,
                                    cols.ctypes.data, rows.size, float(alpha), float(beta),
                                    c_old.ctypes.data if c_old is not None else None,
                                    bias.ctypes.data if bias is not None else None,
                                    int(bool(relu)), out.ctypes.data)
    return out


def trmm(a: np.ndarray, b: np.ndarray, alpha: float = 1.0, nthreads: int | None = None) -> np.ndarray:
    """The TRMM page's product C = fp16(alpha·Aᵀ·B), (n, m) float16, for a
    (n, n) whose lower triangle is A (the rest is not read) and b (n, m).
    Arrays are in mathematical orientation; the C code reads them column-major."""
    a = np.asarray(a, dtype=np.float16)
    b = np.asarray(b, dtype=np.float16)
    n = a.shape[0]
    if a.shape != (n, n) or b.ndim != 2 or b.shape[0] != n:
        raise ValueError("a must be (n, n) and b (n, m)")
    m = b.shape[1]
    a_col = np.ascontiguousarray(a.T)      # column c of A is row c here: A(r, c) at [c*n + r]
    b_col = np.ascontiguousarray(b.T)
    c_col = np.empty((m, n), dtype=np.float16)
    rc = _load().oracle_trmm(a_col.ctypes.data, n, b_col.ctypes.data, n, c_col.ctypes.data, n, n, m,
                             float(alpha), _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_trmm could not allocate its thread bookkeeping")
    return np.ascontiguousarray(c_col.T)


def trsm(a: np.ndarray, b: np.ndarray, alpha: float = 1.0, nthreads: int | None = None) -> np.ndarray:
    """The TRMM page's triangular solve: X (n, m) float16 with Aᵀ·X = alpha·B,
    for a (n, n) whose lower triangle is A (the rest is not read) and b (n, m),
    in mathematical orientation; FP64 back substitution, one rounding."""
    a = np.asarray(a, dtype=np.float16)
    b = np.asarray(b, dtype=np.float16)
    n = a.shape[0]
    if a.shape != (n, n) or b.ndim != 2 or b.shape[0] != n:
        raise ValueError("a must be (n, n) and b (n, m)")
    m = b.shape[1]
    a_col = np.ascontiguousarray(a.T)
    b_col = np.ascontiguousarray(b.T)
    x_col = np.empty((m, n), dtype=np.float16)
    rc = _load().oracle_trsm(a_col.ctypes.data, n, b_col.ctypes.data, n, x_col.ctypes.data, n, n, m,
                             float(alpha), _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_trsm could not allocate its work space")
    return np.ascontiguousarray(x_col.T)


def trsm_n(a: np.ndarray, b: np.ndarray, alpha: float = 1.0, nthreads: int | None = None) -> np.ndarray:
    """The solve in the TRMM page's literal orientation (§2.3, X = A\\B):
    X (n, m) float16 with A·X = alpha·B, A the lower triangle of a (n, n)
    (the rest is not read), b (n, m), in mathematical orientation; FP64
    forward substitution, one rounding."""
    a = np.asarray(a, dtype=np.float16)
    b = np.asarray(b, dtype=np.float16)
    n = a.shape[0]
    if a.shape != (n, n) or b.ndim != 2 or b.shape[0] != n:
        raise ValueError("a must be (n, n) and b (n, m)")
    m = b.shape[1]
    a_col = np.ascontiguousarray(a.T)
    b_col = np.ascontiguousarray(b.T)
    x_col = np.empty((m, n), dtype=np.float16)
    rc = _load().oracle_trsm_n(a_col.ctypes.data, n, b_col.ctypes.data, n, x_col.ctypes.data, n, n, m,
                               float(alpha), _threads(nthreads))
    if rc != 0:
        raise MemoryError("oracle_trsm_n could not allocate its work space")
    return np.ascontiguousarray(x_col.T)


def fp16_to_double(bits: int) -> float:
    """Decodes one binary16 bit pattern."""
    return _load().oracle_fp16_to_double(bits & 0xFFFF)


def double_to_fp16(x: float) -> int:
    """Rounds one double to the nearest binary16 (ties to even); returns the bits."""
    return int(_load().oracle_double_to_fp16(float(x)))
