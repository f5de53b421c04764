"""The C-ABI boundary on the host: the library loads, exports every symbol the
header declares, and its host-only logic (argument checks, path selection,
status text) behaves as documented. No computing call is made here."""

import ctypes
import os
import re
import shutil

import pytest

import tensor_core_dense_fp16_gb300 as tc
from tensor_core_dense_fp16_gb300 import build as tcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hgemm.h")


@pytest.fixture(scope="module")
def lib():
    tcbuild.build()
    return tc.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"HGEMM_API\s+[\w\s\*]+?\b(hgemm\w*)\s*\(", text)


def declared_constants():
    text = open(HEADER, encoding="utf-8").read()
    out = {}
    for name, val in re.findall(r"#define\s+(HGEMM_(?:OK|ERR_\w+|PATH_\w+|TRSM_(?:AUTO|SUBSTITUTION|RECURSIVE|CHAIN\w*)))\s+\(?(-?\d+)\)?", text):
        out[name] = int(val)
    return out


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"hgemm", "hgemm_host", "hgemm_select_path", "hgemm_force_path",
            "hgemm_device_status", "hgemm_last_cuda_error", "hgemm_status_string",
            "hgemm_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        # and the binding exposes the same name
        assert callable(getattr(tc, n)), n


def test_binding_constants_match_header():
    consts = declared_constants()
    assert len(consts) >= 11
    for name, val in consts.items():
        assert getattr(tc, name) == val, name


def test_trsm_schedule_hooks(lib):
    """The schedule override takes the settable HGEMM_TRSM_* values and
    nothing else; the last schedule is host state."""
    try:
        for bad in (-1, tc.HGEMM_TRSM_SUBSTITUTION, 6, 99):
            with pytest.raises(tc.HgemmError) as err:
                tc.hgemm_force_trsm_schedule(bad)
            assert err.value.status == tc.HGEMM_ERR_INVALID_ARG
        for ok in (tc.HGEMM_TRSM_RECURSIVE, tc.HGEMM_TRSM_CHAIN, tc.HGEMM_TRSM_CHAIN_FUSED,
                   tc.HGEMM_TRSM_CHAIN_SPLIT, tc.HGEMM_TRSM_AUTO):
            tc.hgemm_force_trsm_schedule(ok)
    finally:
        tc.hgemm_force_trsm_schedule(tc.HGEMM_TRSM_AUTO)
    assert tc.hgemm_trsm_last_schedule() in (0, tc.HGEMM_TRSM_SUBSTITUTION, tc.HGEMM_TRSM_RECURSIVE,
                                             tc.HGEMM_TRSM_CHAIN_FUSED, tc.HGEMM_TRSM_CHAIN_SPLIT)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        s = tc.hgemm_status_string(code)
        assert s and s != "unknown status"
    assert tc.hgemm_status_string(-99) == "unknown status"
    assert tc.hgemm_version() == (0, 1)


A16, B16, C16 = 0x10000000, 0x20000000, 0x30000000  # 16-byte aligned, disjoint


def test_path_selection(lib):
    sel = tc.hgemm_select_path
    assert sel(A16, B16, C16, 0, 5, 5) == tc.HGEMM_PATH_NONE
    assert sel(A16, B16, C16, 5, 0, 5) == tc.HGEMM_PATH_NONE
    assert sel(A16, B16, C16, 4, 8, 0) == tc.HGEMM_PATH_ZERO
    # enough 256x512 tiles for every CTA pair: wide pair tiles
    assert sel(A16, B16, C16, 8192, 8192, 8192) == tc.HGEMM_PATH_TC_WIDE
    assert sel(A16, B16, C16, 4096, 4096, 4096) == tc.HGEMM_PATH_TC_WIDE
    # fewer: 256x256 pair tiles
    assert sel(A16, B16, C16, 2048, 2048, 2048) == tc.HGEMM_PATH_TC_PAIR
    assert sel(A16, B16, C16, 4096, 2048, 1024) == tc.HGEMM_PATH_TC_PAIR
    # few tiles and a long K (48 K blocks or more): split K over clusters of pairs
    assert sel(A16, B16, C16, 4096, 256, 4096) == tc.HGEMM_PATH_SKINNY
    assert sel(A16, B16, C16, 512, 512, 3072) == tc.HGEMM_PATH_SKINNY
    # a shorter K is not worth the exchange of partial sums; an output that
    # one wave of 128x64 tiles covers (152 on a GB300) takes one CTA per tile
    assert sel(A16, B16, C16, 1000, 1000, 1000) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 256, 256, 256) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 4096, 256, 2048) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 19 * 128, 8 * 64, 1024) == tc.HGEMM_PATH_TC_NARROW   # 152 tiles
    # one more tile row: 256-wide pair tiles, cut into 128- or 64-column parts
    assert sel(A16, B16, C16, 20 * 128, 8 * 64, 1024) == tc.HGEMM_PATH_TC_PAIR
    assert sel(A16, B16, C16, 4096, 512, 2048) == tc.HGEMM_PATH_TC_PAIR
    # more than half of the pairs busy without splitting: no split
    assert sel(A16, B16, C16, 256 * 39, 256, 4096) == tc.HGEMM_PATH_TC_PAIR
    # too little K to split: one K block
    assert sel(A16, B16, C16, 4096, 256, 64) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 8192, 256, 64) == tc.HGEMM_PATH_TC_PAIR
    assert sel(A16, B16, C16, 128, 256, 64) == tc.HGEMM_PATH_TC_NARROW
    # 128 rows or fewer with many tiles: one CTA per 128x256 tile
    assert sel(A16, B16, C16, 128, 16384, 4096) == tc.HGEMM_PATH_TC
    # TMA needs 16-byte row pitches and 16-byte base addresses
    assert sel(A16, B16, C16, 64, 64, 1001) == tc.HGEMM_PATH_GENERIC
    assert sel(A16, B16, C16, 64, 1001, 64) == tc.HGEMM_PATH_GENERIC
    assert sel(A16 + 2, B16, C16, 64, 64, 64) == tc.HGEMM_PATH_GENERIC
    assert sel(A16, B16 + 8, C16, 64, 64, 64) == tc.HGEMM_PATH_GENERIC
    assert sel(A16, B16, C16 + 4, 64, 64, 64) == tc.HGEMM_PATH_GENERIC
    # M is free: any M works with TMA
    assert sel(A16, B16, C16, 1001, 64, 64) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 1200, 1024, 64) == tc.HGEMM_PATH_TC_PAIR
    assert sel(A16, B16, C16, 1, 64, 64) == tc.HGEMM_PATH_TC_NARROW
    assert sel(A16, B16, C16, 1, 10240, 64) == tc.HGEMM_PATH_TC
    assert sel(A16, B16, C16, 1, 64, 4096) == tc.HGEMM_PATH_SKINNY


def test_forced_paths(lib):
    try:
        tc.hgemm_force_path(tc.HGEMM_PATH_GENERIC)
        assert tc.hgemm_select_path(A16, B16, C16, 256, 256, 256) == tc.HGEMM_PATH_GENERIC
        tc.hgemm_force_path(tc.HGEMM_PATH_TC)
        assert tc.hgemm_select_path(A16, B16, C16, 256, 256, 256) == tc.HGEMM_PATH_TC
        tc.hgemm_force_path(tc.HGEMM_PATH_TC_NARROW)
        assert tc.hgemm_select_path(A16, B16, C16, 8192, 8192, 8192) == tc.HGEMM_PATH_TC_NARROW
        tc.hgemm_force_path(tc.HGEMM_PATH_TC_PAIR)
        assert tc.hgemm_select_path(A16, B16, C16, 64, 256, 256) == tc.HGEMM_PATH_TC_PAIR
        tc.hgemm_force_path(tc.HGEMM_PATH_TC_WIDE)
        assert tc.hgemm_select_path(A16, B16, C16, 256, 256, 256) == tc.HGEMM_PATH_TC_WIDE
        tc.hgemm_force_path(tc.HGEMM_PATH_SKINNY)
        assert tc.hgemm_select_path(A16, B16, C16, 8192, 8192, 8192) == tc.HGEMM_PATH_TC_PAIR
        assert tc.hgemm_select_path(A16, B16, C16, 512, 512, 512) == tc.HGEMM_PATH_SKINNY
        # a single K block cannot be split
        assert tc.hgemm_select_path(A16, B16, C16, 512, 512, 64) == tc.HGEMM_PATH_TC_PAIR
        # a forced TMA path still needs TMA-able operands
        assert tc.hgemm_select_path(A16, B16, C16, 256, 256, 255) == tc.HGEMM_PATH_GENERIC
        with pytest.raises(tc.HgemmError):
            tc.hgemm_force_path(77)
    finally:
        tc.hgemm_force_path(-1)
    assert tc.hgemm_select_path(A16, B16, C16, 256, 256, 256) == tc.HGEMM_PATH_TC_NARROW


def test_forced_split_configuration(lib):
    for bad in [(1, 256), (5, 256), (3, 128), (2, 64), (0, 256)]:
        with pytest.raises(tc.HgemmError):
            tc.hgemm_force_split(*bad)
    try:
        tc.hgemm_force_path(tc.HGEMM_PATH_SKINNY)
        for good in [(2, 128), (2, 256), (3, 256), (4, 256)]:
            tc.hgemm_force_split(*good)
            assert tc.hgemm_select_path(A16, B16, C16, 4096, 256, 4096) == tc.HGEMM_PATH_SKINNY
    finally:
        tc.hgemm_force_split(0, 0)
        tc.hgemm_force_path(-1)


def test_fused_argument_checks(lib):
    """hgemm_ex rejects a misaligned bias and a bias that overlaps C before any
    device work (fake addresses)."""
    lib_ = tc.load()
    rc = lib_.hgemm_ex(A16, B16, C16, 4, 8, 8, 1.0, 0.0, 0x40000001, 0, None)
    assert rc == tc.HGEMM_ERR_INVALID_ARG
    rc = lib_.hgemm_ex(A16, B16, C16, 4, 8, 8, 1.0, 1.0, C16 + 16, 1, None)
    assert rc == tc.HGEMM_ERR_ALIAS
    rc = lib_.hgemm_ex(A16, B16, C16, -1, 8, 8, 1.0, 1.0, None, 0, None)
    assert rc == tc.HGEMM_ERR_INVALID_ARG
    # empty output: nothing to do, no device needed
    assert lib_.hgemm_ex(A16, B16, C16, 0, 8, 8, 2.0, 1.0, 0x40000000, 1, None) == tc.HGEMM_OK


def test_strided_argument_checks(lib):
    lib_ = tc.load()
    # pitches shorter than a row
    assert lib_.hgemm_strided(A16, 7, B16, 8, C16, 8, 4, 8, 8, 1.0, 0.0, None, 0, None) == tc.HGEMM_ERR_INVALID_ARG
    assert lib_.hgemm_strided(A16, 8, B16, 7, C16, 8, 4, 8, 8, 1.0, 0.0, None, 0, None) == tc.HGEMM_ERR_INVALID_ARG
    assert lib_.hgemm_strided(A16, 8, B16, 8, C16, 7, 4, 8, 8, 1.0, 0.0, None, 0, None) == tc.HGEMM_ERR_INVALID_ARG
    # C's span (3 rows of pitch 1024) reaches A
    assert lib_.hgemm_strided(C16 + 2 * 2048, 8, B16, 8, C16, 1024, 3, 8, 8, 1.0, 0.0, None, 0,
                              None) == tc.HGEMM_ERR_ALIAS
    # a huge pitch that would overflow the span
    assert lib_.hgemm_strided(A16, 1 << 41, B16, 8, C16, 8, 4, 8, 8, 1.0, 0.0, None, 0,
                              None) == tc.HGEMM_ERR_INVALID_ARG
    # nothing to do
    assert lib_.hgemm_strided(A16, 8, B16, 8, C16, 8, 0, 8, 8, 1.0, 0.0, None, 0, None) == tc.HGEMM_OK


def test_trmm_argument_checks(lib):
    lib_ = tc.load()
    n, m = 64, 8
    ok = dict(A=A16, lda=n, B=B16, ldb=n, C=C16, ldc=n)
    def call(**kw):
        a = {**ok, **kw}
        return lib_.hgemm_trmm(a["A"], a["lda"], a["B"], a["ldb"], a["C"], a["ldc"], kw.get("n", n),
                               kw.get("m", m), 1.0, None)
    assert call(n=tc.HGEMM_TRMM_MAX_N + 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(n=-1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(lda=n - 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(ldc=n - 8) == tc.HGEMM_ERR_INVALID_ARG
    assert call(A=None) == tc.HGEMM_ERR_INVALID_ARG
    assert call(B=B16 + 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(C=A16 + 2 * 10) == tc.HGEMM_ERR_ALIAS     # C inside A's span
    assert call(n=0) == tc.HGEMM_OK and call(m=0) == tc.HGEMM_OK


def test_trsm_argument_checks(lib):
    lib_ = tc.load()
    n, m = 64, 8
    ok = dict(A=A16, lda=n, B=B16, ldb=n, X=C16, ldx=n)
    def call(**kw):
        a = {**ok, **kw}
        return lib_.hgemm_trsm(a["A"], a["lda"], a["B"], a["ldb"], a["X"], a["ldx"], kw.get("n", n),
                               kw.get("m", m), 1.0, None)
    assert call(n=-1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(m=-1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(n=tc.HGEMM_MAX_DIM + 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(lda=n - 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(ldb=n - 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(ldx=n - 8) == tc.HGEMM_ERR_INVALID_ARG
    assert call(A=None) == tc.HGEMM_ERR_INVALID_ARG
    assert call(X=C16 + 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(X=A16 + 2 * 10) == tc.HGEMM_ERR_ALIAS     # X inside A's span
    assert call(X=B16 + 2 * 8) == tc.HGEMM_ERR_ALIAS      # X overlaps B, not in place
    assert call(X=B16, ldx=n + 8) == tc.HGEMM_ERR_ALIAS   # X = B with another pitch
    assert call(n=0) == tc.HGEMM_OK and call(m=0) == tc.HGEMM_OK


def test_trsm_workspace_argument_checks(lib):
    """hgemm_trsm_ws and hgemm_trsm_noalloc check their arguments on the host
    before any device work: workspace size per diagonal block of order ≤ 512,
    a missing, short or misaligned workspace, one overlapping an operand, and
    a triangle beyond the fixed array."""
    lib_ = tc.load()
    assert tc.hgemm_trsm_workspace_size(0) == 0
    assert tc.hgemm_trsm_workspace_size(-5) == 0
    # 512 KiB per diagonal block of order <= 512, one spare block, 4 KiB of synchronisation words
    assert tc.hgemm_trsm_workspace_size(512) == 2 * 2 * 512 * 512 + 4096
    assert tc.hgemm_trsm_workspace_size(513) == 3 * 2 * 512 * 512 + 4096
    assert tc.hgemm_trsm_workspace_size(8192) == 17 * 2 * 512 * 512 + 4096 == tc.HGEMM_TRSM_NOALLOC_MAX_BYTES
    assert tc.hgemm_trsm_workspace_size(8193) > tc.HGEMM_TRSM_NOALLOC_MAX_BYTES
    n, m = 64, 8
    need = tc.hgemm_trsm_workspace_size(n)
    W16 = 0x50000000
    ok = dict(A=A16, lda=n, B=B16, ldb=n, X=C16, ldx=n, W=W16, bytes=need)
    def call(**kw):
        a = {**ok, **kw}
        return lib_.hgemm_trsm_ws(a["A"], a["lda"], a["B"], a["ldb"], a["X"], a["ldx"], kw.get("n", n),
                                  kw.get("m", m), 1.0, a["W"], a["bytes"], None)
    assert call(W=None) == tc.HGEMM_ERR_INVALID_ARG
    # the inverses alone (an older workspace size) are still accepted; less is not
    assert call(bytes=need - 4096 - 2 * 512 * 512 - 1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(W=W16 + 8) == tc.HGEMM_ERR_INVALID_ARG
    assert call(W=A16) == tc.HGEMM_ERR_ALIAS
    assert call(W=C16 - 16) == tc.HGEMM_ERR_ALIAS
    assert call(n=-1) == tc.HGEMM_ERR_INVALID_ARG
    assert call(n=0) == tc.HGEMM_OK and call(m=0) == tc.HGEMM_OK
    big = 8193
    assert lib_.hgemm_trsm_noalloc(A16, big, B16, big, C16, big, big, 1, 1.0, None) == tc.HGEMM_ERR_INVALID_ARG
    assert lib_.hgemm_trsm_noalloc(A16, n, B16, n, C16, n, -1, m, 1.0, None) == tc.HGEMM_ERR_INVALID_ARG
    assert lib_.hgemm_trsm_noalloc(A16, n, B16, n, C16, n, 0, m, 1.0, None) == tc.HGEMM_OK


def test_layout_argument_checks(lib):
    lib_ = tc.load()
    def call(a_layout=0, b_layout=0, lda=64, ldb=64, ldc=64, M=16, N=64, K=64, C=C16):
        return lib_.hgemm_layout(a_layout, b_layout, A16, lda, B16, ldb, C, ldc, M, N, K, 1.0, 0.0,
                                 None, 0, None)
    assert call(a_layout=2) == tc.HGEMM_ERR_INVALID_ARG
    assert call(b_layout=-1) == tc.HGEMM_ERR_INVALID_ARG
    # the pitch must cover a stored row: K for A row-major, M for A column-major,
    # K for B column-major, N for B row-major
    assert call(lda=63) == tc.HGEMM_ERR_INVALID_ARG
    assert call(a_layout=1, lda=15) == tc.HGEMM_ERR_INVALID_ARG
    assert call(ldb=63) == tc.HGEMM_ERR_INVALID_ARG
    assert call(b_layout=1, N=72, ldb=64, ldc=72) == tc.HGEMM_ERR_INVALID_ARG
    # spans follow the layout: A column-major is K rows of lda
    assert call(a_layout=1, lda=16, C=A16 + 2 * 16 * 63) == tc.HGEMM_ERR_ALIAS
    assert call(M=0) == tc.HGEMM_OK and call(a_layout=1, b_layout=1, N=0, lda=16) == tc.HGEMM_OK


def test_invalid_arguments_rejected_before_any_device_work(lib):
    bad = [
        (A16, B16, C16, -1, 4, 4),
        (A16, B16, C16, 4, -1, 4),
        (A16, B16, C16, 4, 4, -1),
        (A16, B16, C16, 1 << 31, 4, 4),
        (A16, B16, C16, 4, 4, 1 << 40),
        (None, B16, C16, 4, 4, 4),
        (A16, None, C16, 4, 4, 4),
        (A16, B16, None, 4, 4, 4),
        (A16, B16, C16, (1 << 31) - 1, (1 << 31) - 1, 8),  # M*N elements >= 2^61
        (A16 + 1, B16, C16, 4, 4, 4),  # FP16 pointers must be 2-byte aligned
        (A16, B16 + 3, C16, 4, 4, 4),
        (A16, B16, C16 + 5, 4, 4, 4),
    ]
    for args in bad:
        assert lib.hgemm(*args, None) == tc.HGEMM_ERR_INVALID_ARG, args
        assert lib.hgemm_select_path(*args) == tc.HGEMM_ERR_INVALID_ARG, args
    # NULL operands are fine when their size is zero
    assert lib.hgemm_select_path(None, None, None, 0, 0, 0) == tc.HGEMM_PATH_NONE
    assert lib.hgemm_select_path(None, None, C16, 4, 4, 0) == tc.HGEMM_PATH_ZERO


def test_alias_detection(lib):
    M, N, K = 64, 64, 64
    a_bytes = M * K * 2
    # C overlapping the tail of A
    assert lib.hgemm_select_path(A16, B16, A16 + a_bytes - 2, M, N, K) == tc.HGEMM_ERR_ALIAS
    assert lib.hgemm(A16, B16, A16 + a_bytes - 2, M, N, K, None) == tc.HGEMM_ERR_ALIAS
    # C overlapping the head of B
    assert lib.hgemm_select_path(A16, B16, B16 - 16, M, N, K) == tc.HGEMM_ERR_ALIAS
    # adjacent but disjoint is fine
    assert lib.hgemm_select_path(A16, B16, A16 + a_bytes, M, N, K) == tc.HGEMM_PATH_TC_NARROW
    # A and B may alias each other (both are read-only)
    assert lib.hgemm_select_path(A16, A16, C16, M, N, K) == tc.HGEMM_PATH_TC_NARROW


def test_binding_type_checks():
    torch = pytest.importorskip("torch")
    a = torch.zeros(4, 4, dtype=torch.float32)
    with pytest.raises(TypeError):
        tc.hgemm(a, a, a, 4, 4, 4, stream=0)
    h = torch.zeros(4, 4, dtype=torch.float16)
    with pytest.raises(ValueError):
        tc.hgemm(h, h, h, 4, 4, 4, stream=0)  # host tensors for a device call


def _cuda_include_dir():
    nvcc = shutil.which("nvcc")
    roots = [os.path.dirname(os.path.dirname(nvcc))] if nvcc else []
    roots += [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]
    for r in roots:
        if r and os.path.exists(os.path.join(r, "include", "cuda_runtime_api.h")):
            return os.path.join(r, "include")
    return None


def test_header_is_a_c_interface(lib, tmp_path):
    """A plain C11 program (gcc, pedantic, warnings as errors) includes the
    header, takes the address of every function it declares, links against
    the library and calls the host-only entry points; their answers match
    the binding's. Nothing of C++ leaks through the boundary."""
    gcc, inc = shutil.which("gcc"), _cuda_include_dir()
    if gcc is None or inc is None:
        pytest.skip("gcc or the CUDA runtime headers are not available")
    names = declared_functions()
    src = ["#include <stdio.h>", '#include "hgemm.h"', "typedef void (*fn_t)(void);",
           "static const fn_t fns[] = {"]
    src += [f"  (fn_t)&{n}," for n in names]
    src += ["};",
            "int main(void) {",
            '  printf("%d\\n", (int)(sizeof(fns) / sizeof(fns[0])));',
            '  printf("%d\\n", hgemm_version());',
            '  printf("%s\\n", hgemm_status_string(HGEMM_ERR_ALIAS));',
            '  printf("%zu\\n", hgemm_trsm_workspace_size(8192));',
            f'  printf("%d\\n", hgemm_select_path((const void *){A16:#x}, (const void *){B16:#x}, '
            f'(const void *){C16:#x}, 4096, 256, 4096));',
            f'  printf("%d\\n", hgemm_select_path((const void *){A16:#x}, (const void *){B16:#x}, '
            f'(const void *){A16:#x}, 64, 64, 64));',
            "  return 0;",
            "}"]
    c_file = tmp_path / "consumer.c"
    c_file.write_text("\n".join(src) + "\n")
    libdir = os.path.dirname(tc.library_path())
    exe = tmp_path / "consumer"
    import subprocess
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), "-I", inc, str(c_file), "-L", libdir, "-lhgemm",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert int(out[0]) == len(names)
    assert int(out[1]) == lib.hgemm_version()
    assert out[2] == tc.hgemm_status_string(tc.HGEMM_ERR_ALIAS)
    assert int(out[3]) == tc.hgemm_trsm_workspace_size(8192)
    assert int(out[4]) == tc.hgemm_select_path(A16, B16, C16, 4096, 256, 4096) == tc.HGEMM_PATH_SKINNY
    assert int(out[5]) == tc.HGEMM_ERR_ALIAS
