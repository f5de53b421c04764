"""Python binding of libhgemm.so, the GB300 FP16 tensor-core GEMM C = A·B.

Argument marshalling only: every step of the product runs in the library's
CUDA kernels (see ``include/hgemm.h`` for the contract). Functions carry the
C names. Matrices may be given as torch tensors (their ``data_ptr()`` is
passed), numpy arrays (host memory, for ``hgemm_host``) or raw integer
addresses. Streams may be a ``torch.cuda.Stream``, a raw handle, or None for
torch's current stream.

Layouts, as in "Nvidia Tensor Core-MMA PTX编程入门", §4 示例: A is M×K
row-major, B is K×N column-major (pass it as an (N, K) row-major array whose
row j is column j of B), C is M×N row-major; all FP16.

If the shared library has not been built, every call raises: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "HGEMM_OK", "HGEMM_ERR_INVALID_ARG", "HGEMM_ERR_ALIAS", "HGEMM_ERR_UNSUPPORTED_DEVICE",
    "HGEMM_ERR_CUDA", "HGEMM_ERR_TIMEOUT", "HGEMM_ERR_DEBUG_CHECK", "hgemm_debug_build", "hgemm_debug_code",
    "hgemm_debug_selftest", "HGEMM_PATH_NONE", "HGEMM_PATH_ZERO",
    "HGEMM_PATH_TC", "HGEMM_PATH_SKINNY", "HGEMM_PATH_GENERIC", "HGEMM_PATH_TC_PAIR",
    "HGEMM_PATH_TC_WIDE", "HGEMM_PATH_TC_NARROW", "HGEMM_MAX_DIM",
    "HgemmError", "library_path", "load", "hgemm", "hgemm_host", "hgemm_select_path",
    "hgemm_force_path", "hgemm_device_status", "hgemm_last_cuda_error",
    "hgemm_status_string", "hgemm_version", "hgemm_set_wait_timeout", "hgemm_debug_inject",
    "hgemm_force_split", "hgemm_launch_floor", "hgemm_ex", "hgemm_strided", "hgemm_trmm", "hgemm_trsm", "hgemm_trsm_ws", "hgemm_trsm_workspace_size", "hgemm_trsm_noalloc", "hgemm_trsm_op", "HGEMM_OP_N", "HGEMM_OP_T", "hgemm_layout", "HGEMM_TRMM_MAX_N", "HGEMM_TRSM_NOALLOC_MAX_BYTES",
    "hgemm_force_trsm_schedule", "hgemm_trsm_last_schedule", "HGEMM_TRSM_AUTO", "HGEMM_TRSM_SUBSTITUTION",
    "HGEMM_TRSM_RECURSIVE", "HGEMM_TRSM_CHAIN", "HGEMM_TRSM_CHAIN_FUSED", "HGEMM_TRSM_CHAIN_SPLIT",
    "HGEMM_A_ROW_MAJOR", "HGEMM_A_COL_MAJOR", "HGEMM_B_COL_MAJOR", "HGEMM_B_ROW_MAJOR",
    "HGEMM_INJECT_NONE", "HGEMM_INJECT_DROP_ARRIVAL", "matmul",
]

HGEMM_OK = 0
HGEMM_ERR_INVALID_ARG = -1
HGEMM_ERR_ALIAS = -2
HGEMM_ERR_UNSUPPORTED_DEVICE = -3
HGEMM_ERR_CUDA = -4
HGEMM_ERR_TIMEOUT = -5
HGEMM_ERR_DEBUG_CHECK = -6
HGEMM_TRMM_MAX_N = 16384
HGEMM_TRSM_NOALLOC_MAX_BYTES = (17 << 19) + 4096
HGEMM_TRSM_AUTO = 0
HGEMM_TRSM_SUBSTITUTION = 1
HGEMM_TRSM_RECURSIVE = 2
HGEMM_TRSM_CHAIN = 3
HGEMM_TRSM_CHAIN_FUSED = 4
HGEMM_TRSM_CHAIN_SPLIT = 5
HGEMM_OP_N = 0
HGEMM_OP_T = 1
HGEMM_A_ROW_MAJOR = 0
HGEMM_A_COL_MAJOR = 1
HGEMM_B_COL_MAJOR = 0
HGEMM_B_ROW_MAJOR = 1

HGEMM_PATH_NONE = 0
HGEMM_PATH_ZERO = 1
HGEMM_PATH_TC = 2
HGEMM_PATH_SKINNY = 3
HGEMM_PATH_GENERIC = 4
HGEMM_PATH_TC_PAIR = 5
HGEMM_PATH_TC_WIDE = 6
HGEMM_PATH_TC_NARROW = 7

HGEMM_MAX_DIM = 0x7FFFFFFF

HGEMM_INJECT_NONE = 0
HGEMM_INJECT_DROP_ARRIVAL = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
# HGEMM_LIBRARY_VARIANT=debug: the -DHGEMM_DEBUG build with device-side checks
_LIB_PATH = (os.path.join(_HERE, "_build", "debug", "libhgemm.so")
             if os.environ.get("HGEMM_LIBRARY_VARIANT") == "debug"
             else os.path.join(_HERE, "_build", "libhgemm.so"))
_lib = None


class HgemmError(RuntimeError):
    """A negative status from libhgemm."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {hgemm_status_string(status)} (status {status})"
        if status == HGEMM_ERR_CUDA:
            msg += f", cudaError {hgemm_last_cuda_error()}"
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load():
    """Loads libhgemm.so (built by tensor_core_dense_fp16_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.hgemm.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    lib.hgemm.restype = i32
    lib.hgemm_ex.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_float, ctypes.c_float, vp,
                             i32, vp]
    lib.hgemm_ex.restype = i32
    lib.hgemm_strided.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, ctypes.c_float,
                                  ctypes.c_float, vp, i32, vp]
    lib.hgemm_strided.restype = i32
    lib.hgemm_trmm.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ctypes.c_float, vp]
    lib.hgemm_trmm.restype = i32
    lib.hgemm_trsm.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ctypes.c_float, vp]
    lib.hgemm_trsm.restype = i32
    lib.hgemm_trsm_ws.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ctypes.c_float, vp, ctypes.c_size_t, vp]
    lib.hgemm_trsm_ws.restype = i32
    lib.hgemm_trsm_workspace_size.argtypes = [i64]
    lib.hgemm_trsm_workspace_size.restype = ctypes.c_size_t
    lib.hgemm_trsm_op.argtypes = [i32, vp, i64, vp, i64, vp, i64, i64, i64, ctypes.c_float, vp,
                                  ctypes.c_size_t, vp]
    lib.hgemm_trsm_op.restype = i32
    lib.hgemm_trsm_noalloc.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, ctypes.c_float, vp]
    lib.hgemm_trsm_noalloc.restype = i32
    lib.hgemm_layout.argtypes = [i32, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_float, vp, i32, vp]
    lib.hgemm_layout.restype = i32
    lib.hgemm_host.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp]
    lib.hgemm_host.restype = i32
    lib.hgemm_select_path.argtypes = [vp, vp, vp, i64, i64, i64]
    lib.hgemm_select_path.restype = i32
    lib.hgemm_force_path.argtypes = [i32]
    lib.hgemm_force_path.restype = i32
    lib.hgemm_device_status.argtypes = [vp]
    lib.hgemm_device_status.restype = i32
    lib.hgemm_last_cuda_error.argtypes = []
    lib.hgemm_last_cuda_error.restype = i32
    lib.hgemm_status_string.argtypes = [i32]
    lib.hgemm_status_string.restype = ctypes.c_char_p
    lib.hgemm_version.argtypes = []
    lib.hgemm_version.restype = i32
    lib.hgemm_set_wait_timeout.argtypes = [ctypes.c_ulonglong]
    lib.hgemm_set_wait_timeout.restype = i32
    lib.hgemm_debug_inject.argtypes = [i32]
    lib.hgemm_debug_inject.restype = i32
    lib.hgemm_force_split.argtypes = [i32, i32]
    lib.hgemm_force_split.restype = i32
    lib.hgemm_launch_floor.argtypes = [i32, vp]
    lib.hgemm_launch_floor.restype = i32
    lib.hgemm_force_trsm_schedule.argtypes = [i32]
    lib.hgemm_force_trsm_schedule.restype = i32
    for name in ("hgemm_debug_build", "hgemm_debug_code", "hgemm_debug_selftest", "hgemm_trsm_last_schedule"):
        getattr(lib, name).argtypes = []
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


# ----------------------------------------------------------------- marshalling

def _ptr(x) -> int | None:
    """Address of a torch tensor, numpy array, ctypes object or integer."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):          # torch.Tensor
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):            # numpy.ndarray
        return int(x.ctypes.data)
    if isinstance(x, ctypes.c_void_p):
        return x.value
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _check_tensor(x, name: str, on_device: bool | None):
    """dtype and contiguity checks for torch tensors and numpy arrays."""
    if hasattr(x, "data_ptr") and hasattr(x, "dtype"):
        import torch
        if x.dtype != torch.float16:
            raise TypeError(f"{name} must be torch.float16, got {x.dtype}")
        if not x.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if on_device is True and not x.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if on_device is False and x.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    elif hasattr(x, "ctypes") and hasattr(x, "dtype"):
        import numpy as np
        if x.dtype != np.float16:
            raise TypeError(f"{name} must be float16, got {x.dtype}")
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{name} must be C-contiguous")
        if on_device is True:
            raise ValueError(f"{name} must be device memory, got a numpy array")


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    raise TypeError(f"cannot use {type(stream).__name__} as a CUDA stream")


def _raise_on(status: int, where: str) -> int:
    if status < 0:
        raise HgemmError(status, where)
    return status


# --------------------------------------------------------------------- the ABI

def hgemm(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """C = A·B on `stream` (enqueued; synchronise the stream to read C)."""
    for x, n in ((A, "A"), (B, "B"), (C, "C")):
        _check_tensor(x, n, True)
    _raise_on(load().hgemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream)), "hgemm")


def hgemm_ex(A, B, C, M: int, N: int, K: int, alpha: float = 1.0, beta: float = 0.0, bias=None,
             relu: bool = False, stream=None) -> None:
    """C = f(alpha·A·B + beta·C + bias[j]) on `stream`, f = ReLU if relu (see hgemm.h)."""
    for x, n in ((A, "A"), (B, "B"), (C, "C")):
        _check_tensor(x, n, True)
    if bias is not None:
        _check_tensor(bias, "bias", True)
    _raise_on(load().hgemm_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, float(alpha), float(beta),
                              _ptr(bias), int(bool(relu)), _stream(stream)), "hgemm_ex")


def hgemm_strided(A, lda: int, B, ldb: int, C, ldc: int, M: int, N: int, K: int,
                  alpha: float = 1.0, beta: float = 0.0, bias=None, relu: bool = False,
                  stream=None) -> None:
    """hgemm_ex on sub-matrices with row pitches (see hgemm.h). A, B, C may be
    tensors (their base address is used) or raw integer addresses."""
    _raise_on(load().hgemm_strided(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, M, N, K, float(alpha),
                                   float(beta), _ptr(bias), int(bool(relu)), _stream(stream)),
              "hgemm_strided")


def hgemm_layout(a_layout: int, b_layout: int, A, lda: int, B, ldb: int, C, ldc: int, M: int,
                 N: int, K: int, alpha: float = 1.0, beta: float = 0.0, bias=None,
                 relu: bool = False, stream=None) -> None:
    """hgemm_strided with a storage order per operand (HGEMM_A_* / HGEMM_B_*; see hgemm.h)."""
    _raise_on(load().hgemm_layout(int(a_layout), int(b_layout), _ptr(A), lda, _ptr(B), ldb, _ptr(C),
                                  ldc, M, N, K, float(alpha), float(beta), _ptr(bias),
                                  int(bool(relu)), _stream(stream)), "hgemm_layout")


def hgemm_trmm(A, lda: int, B, ldb: int, C, ldc: int, n: int, m: int, alpha: float = 1.0,
               stream=None) -> None:
    """C = alpha·Aᵀ·B, A lower triangular; column-major operands (see hgemm.h)."""
    _raise_on(load().hgemm_trmm(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, n, m, float(alpha),
                                _stream(stream)), "hgemm_trmm")


def hgemm_trsm(A, lda: int, B, ldb: int, X, ldx: int, n: int, m: int, alpha: float = 1.0,
               stream=None) -> None:
    """Solves Aᵀ·X = alpha·B for X, A lower triangular; column-major operands;
    X may be B itself (same pitch) to solve in place (see hgemm.h)."""
    _raise_on(load().hgemm_trsm(_ptr(A), lda, _ptr(B), ldb, _ptr(X), ldx, n, m, float(alpha),
                                _stream(stream)), "hgemm_trsm")


def hgemm_trsm_noalloc(A, lda: int, B, ldb: int, X, ldx: int, n: int, m: int, alpha: float = 1.0,
                       stream=None) -> None:
    """hgemm_trsm_ws with the library's fixed device workspace instead of one
    from the caller: allocates nothing (for callers that cannot allocate);
    n up to 8192 (see hgemm.h for the set-up on first use and the sharing
    of the workspace between calls)."""
    _raise_on(load().hgemm_trsm_noalloc(_ptr(A), lda, _ptr(B), ldb, _ptr(X), ldx, n, m, float(alpha),
                                        _stream(stream)), "hgemm_trsm_noalloc")


def hgemm_trsm_workspace_size(n: int) -> int:
    """Bytes of device workspace hgemm_trsm_ws uses for a triangle of order n."""
    return int(load().hgemm_trsm_workspace_size(n))


def hgemm_trsm_ws(A, lda: int, B, ldb: int, X, ldx: int, n: int, m: int, alpha: float = 1.0,
                  workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    """hgemm_trsm with a caller-owned device workspace (a tensor or an
    address; its size defaults to the tensor's bytes), see hgemm.h."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _raise_on(load().hgemm_trsm_ws(_ptr(A), lda, _ptr(B), ldb, _ptr(X), ldx, n, m, float(alpha),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream)), "hgemm_trsm_ws")


def hgemm_trsm_op(op: int, A, lda: int, B, ldb: int, X, ldx: int, n: int, m: int, alpha: float = 1.0,
                  workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    """Solves A·X = alpha·B (op = HGEMM_OP_N, the page's literal X = A\\B) or
    Aᵀ·X = alpha·B (HGEMM_OP_T) for X, A lower triangular, column-major
    operands; with an optional workspace as hgemm_trsm_ws takes (see hgemm.h)."""
    if workspace_bytes is None:
        workspace_bytes = (workspace.numel() * workspace.element_size() if hasattr(workspace, "numel")
                           else 0)
    _raise_on(load().hgemm_trsm_op(int(op), _ptr(A), lda, _ptr(B), ldb, _ptr(X), ldx, n, m, float(alpha),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream)), "hgemm_trsm_op")


def hgemm_host(hA, hB, hC, M: int, N: int, K: int, dA, dB, dC, stream=None) -> None:
    """Host operands: H2D copies, the product and the D2H copy, all on `stream`."""
    for x, n in ((hA, "hA"), (hB, "hB"), (hC, "hC")):
        _check_tensor(x, n, False)
    for x, n in ((dA, "dA"), (dB, "dB"), (dC, "dC")):
        _check_tensor(x, n, True)
    _raise_on(load().hgemm_host(_ptr(hA), _ptr(hB), _ptr(hC), M, N, K, _ptr(dA), _ptr(dB),
                                _ptr(dC), _stream(stream)), "hgemm_host")


def hgemm_select_path(A, B, C, M: int, N: int, K: int) -> int:
    """The HGEMM_PATH_* hgemm would take (host logic only; raises on bad args)."""
    return _raise_on(load().hgemm_select_path(_ptr(A), _ptr(B), _ptr(C), M, N, K),
                     "hgemm_select_path")


def hgemm_force_path(path: int) -> None:
    _raise_on(load().hgemm_force_path(path), "hgemm_force_path")


def hgemm_force_trsm_schedule(schedule: int) -> None:
    """Testing aid: HGEMM_TRSM_RECURSIVE keeps solves with a workspace on the
    recursion's launches; HGEMM_TRSM_CHAIN (either plan), HGEMM_TRSM_CHAIN_FUSED
    or HGEMM_TRSM_CHAIN_SPLIT force the one persistent launch; HGEMM_TRSM_AUTO
    chooses."""
    _raise_on(load().hgemm_force_trsm_schedule(schedule), "hgemm_force_trsm_schedule")


def hgemm_trsm_last_schedule() -> int:
    """The HGEMM_TRSM_* schedule of the last solve enqueued on this thread."""
    return int(load().hgemm_trsm_last_schedule())


def hgemm_device_status(stream=None) -> int:
    """Synchronises `stream`; returns HGEMM_OK, HGEMM_ERR_TIMEOUT or (debug
    build) HGEMM_ERR_DEBUG_CHECK; raises otherwise."""
    st = load().hgemm_device_status(_stream(stream))
    if st in (HGEMM_OK, HGEMM_ERR_TIMEOUT, HGEMM_ERR_DEBUG_CHECK):
        return st
    raise HgemmError(st, "hgemm_device_status")


def hgemm_debug_build() -> int:
    return int(load().hgemm_debug_build())


def hgemm_debug_code() -> int:
    return int(load().hgemm_debug_code())


def hgemm_debug_selftest() -> int:
    return int(load().hgemm_debug_selftest())


def hgemm_launch_floor(pair_config: bool = True, stream=None) -> None:
    """Enqueues a kernel that does nothing (the pair kernel's launch
    configuration when pair_config), to time the fixed cost of a launch."""
    _raise_on(load().hgemm_launch_floor(1 if pair_config else 0, _stream(stream)), "hgemm_launch_floor")


def hgemm_last_cuda_error() -> int:
    return int(load().hgemm_last_cuda_error())


def hgemm_status_string(status: int) -> str:
    return load().hgemm_status_string(status).decode()


def hgemm_version() -> tuple[int, int]:
    v = int(load().hgemm_version())
    return v >> 16, v & 0xFFFF


def hgemm_set_wait_timeout(ns: int) -> None:
    """Time limit of every in-kernel wait for later calls (0: default 2 s)."""
    _raise_on(load().hgemm_set_wait_timeout(int(ns)), "hgemm_set_wait_timeout")


def hgemm_debug_inject(what: int) -> None:
    """Testing aid for the watchdog (HGEMM_INJECT_*); see include/hgemm.h."""
    _raise_on(load().hgemm_debug_inject(int(what)), "hgemm_debug_inject")


def hgemm_force_split(split: int, tile_n: int) -> None:
    """Testing aid: the split-K configuration for later calls ((0, 0): automatic)."""
    _raise_on(load().hgemm_force_split(int(split), int(tile_n)), "hgemm_force_split")


def matmul(a, b_cols, out=None, stream=None):
    """Convenience: a (M, K) and b_cols (N, K) CUDA float16 tensors -> (M, N).

    Row j of ``b_cols`` is column j of B. Allocates ``out`` with torch if not
    given (the library itself never allocates)."""
    import torch
    M, K = a.shape
    N, K2 = b_cols.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    elif tuple(out.shape) != (M, N):
        raise ValueError(f"out must be ({M}, {N})")
    hgemm(a, b_cols, out, M, N, K, stream)
    return out
