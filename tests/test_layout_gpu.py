"""hgemm_layout: the product with A stored M×K row-major or K×M (column-major),
and B stored N×K (column-major, as hgemm) or K×N row-major (the CUDA
chapter's layout, "GPU架构与CUDA", 共享内存与分块), against the oracle (GPU
only). The oracle takes A as (M, K) and B as (N, K); the tests lay the same
values out in the requested order on the device."""

import numpy as np
import pytest

import oracle
import synth
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, oracle_threads, to_device, torch_cuda

pytestmark = pytest.mark.gpu

LAYOUTS = [(tc.HGEMM_A_ROW_MAJOR, tc.HGEMM_B_COL_MAJOR), (tc.HGEMM_A_ROW_MAJOR, tc.HGEMM_B_ROW_MAJOR),
           (tc.HGEMM_A_COL_MAJOR, tc.HGEMM_B_COL_MAJOR), (tc.HGEMM_A_COL_MAJOR, tc.HGEMM_B_ROW_MAJOR)]
NAMES = {(0, 0): "A row, B col", (0, 1): "A row, B row", (1, 0): "A col, B col", (1, 1): "A col, B row"}


def stored(x, pad, fill=0.0):
    """x (rows, cols) in a (rows, cols + pad) buffer: row pitch cols + pad."""
    rows, cols = x.shape
    buf = np.full((rows, cols + pad), fill, np.float16)
    buf[:, :cols] = x
    return buf


def run_layout(a, b, a_layout, b_layout, c_old=None, alpha=1.0, beta=0.0, bias=None, relu=False,
               pad=(0, 0, 0), path=None, split=None):
    """a (M, K), b (N, K) in mathematical orientation; returns C (M, N)."""
    torch = torch_cuda()
    M, K = a.shape
    N = b.shape[0]
    a_st = a if a_layout == tc.HGEMM_A_ROW_MAJOR else np.ascontiguousarray(a.T)   # (M,K) or (K,M)
    b_st = b if b_layout == tc.HGEMM_B_COL_MAJOR else np.ascontiguousarray(b.T)   # (N,K) or (K,N)
    a_buf, b_buf = stored(a_st, pad[0]), stored(b_st, pad[1])
    c_buf = stored(c_old if c_old is not None else np.zeros((M, N), np.float16), pad[2], fill=3.0)
    if c_old is None:
        c_buf[:, :N] = np.nan
    da, db, dc = to_device(a_buf), to_device(b_buf), to_device(c_buf)
    dbias = to_device(bias) if bias is not None else None
    if path is not None:
        tc.hgemm_force_path(path)
    if split is not None:
        tc.hgemm_force_split(*split)
    try:
        tc.hgemm_layout(a_layout, b_layout, da, a_buf.shape[1], db, b_buf.shape[1], dc, c_buf.shape[1],
                        M, N, K, alpha, beta, dbias, relu)
    finally:
        tc.hgemm_force_path(-1)
        tc.hgemm_force_split(0, 0)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    out = dc.cpu().numpy()
    assert np.all(out[:, N:] == 3.0), "pitch padding of C was written"
    return out[:, :N]


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1000, 520, 384), (300, 136, 200), (2048, 2048, 2048),
                                   (64, 1024, 4096)])
def test_layout_matches_oracle(layout, M, N, K):
    a, b = synth.operands(M, N, K, seed=M + N + K, kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout), ref, what=f"{NAMES[layout]} {M}x{N}x{K}")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
def test_layout_integer_bit_exact(layout):
    M, N, K = 520, 384, 256
    a, b = synth.operands(M, N, K, seed=77, kind="int")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout), ref, exact=True, what=f"{NAMES[layout]} int")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
@pytest.mark.parametrize("pad", [(8, 16, 8), (3, 5, 1)])
def test_layout_pitches(layout, pad):
    """Padded pitches: multiples of 8 (tensor-core path) and odd ones (the
    generic kernel, which gathers M- or N-contiguous operands)."""
    M, N, K = 333, 200, 150
    a, b = synth.operands(M, N, K, seed=5 + pad[0], kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout, pad=pad), ref, what=f"{NAMES[layout]} pad {pad}")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
@pytest.mark.parametrize("path", [tc.HGEMM_PATH_TC_PAIR, tc.HGEMM_PATH_TC_WIDE], ids=["pair", "wide"])
@pytest.mark.parametrize("M,N,K", [(1000, 520, 384), (513, 1032, 200)])
def test_layout_forced_tensor_core_paths(layout, path, M, N, K):
    """The pair and wide kernels read MN-major tiles, with ragged edges."""
    a, b = synth.operands(M, N, K, seed=M + 3 * N, kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout, path=path), ref, what=f"{NAMES[layout]} path {path}")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
def test_layout_wide_chosen(layout):
    """A shape with a 256×512 tile for every SM pair: the wide kernel, ragged in M and N."""
    M, N, K = 4000, 4104, 1000
    a, b = synth.operands(M, N, K, seed=4000, kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout), ref, what=f"{NAMES[layout]} wide")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
@pytest.mark.parametrize("split", [(2, 128), (2, 256), (3, 256), (4, 256)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_layout_split_k(layout, split):
    """The split-K cluster kernel reads M- and N-contiguous operands too
    (ragged M, K not a multiple of the slices)."""
    M, N, K = 1000, 512, 4000
    a, b = synth.operands(M, N, K, seed=17 + split[0], kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    got = run_layout(a, b, *layout, path=tc.HGEMM_PATH_SKINNY, split=split)
    assert_close(got, ref, what=f"{NAMES[layout]} split {split}")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
def test_layout_skinny_shape(layout):
    """The 4096×256×4096 shape (the TRMM page's update) takes split-K in every layout."""
    M, N, K = 4096, 256, 4096
    a, b = synth.operands(M, N, K, seed=1004, kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout), ref, what=f"{NAMES[layout]} skinny")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
def test_layout_generic_forced(layout):
    M, N, K = 260, 136, 130
    a, b = synth.operands(M, N, K, seed=9, kind="uniform")
    ref = oracle.hgemm(a, b, nthreads=oracle_threads())
    assert_close(run_layout(a, b, *layout, path=tc.HGEMM_PATH_GENERIC), ref,
                 what=f"{NAMES[layout]} generic")


@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: NAMES[l])
def test_layout_fused_epilogue(layout):
    M, N, K = 1000, 520, 384
    a, b = synth.operands(M, N, K, seed=31, kind="uniform")
    rng = np.random.default_rng(31)
    c_old = rng.uniform(-4, 4, size=(M, N)).astype(np.float16)
    bias = rng.uniform(-2, 2, size=N).astype(np.float16)
    ref = oracle.hgemm_ex(a, b, c_old, -1.25, 0.5, bias, True, nthreads=oracle_threads())
    got = run_layout(a, b, *layout, c_old=c_old, alpha=-1.25, beta=0.5, bias=bias, relu=True)
    assert_close(got, ref, what=f"{NAMES[layout]} fused")


@pytest.mark.parametrize("layout", LAYOUTS[1:], ids=lambda l: NAMES[l])
def test_layout_4096_sampled(layout):
    """A 4096-cube (the wide kernel) in the other layouts, sampled rows and
    columns against the oracle's single entries."""
    torch = torch_cuda()
    M = N = K = 4096
    a, b = synth.operands(M, N, K, seed=1234, kind="normal")
    a_l, b_l = layout
    da = to_device(np.ascontiguousarray(a.T) if a_l == tc.HGEMM_A_COL_MAJOR else a)
    db = to_device(np.ascontiguousarray(b.T) if b_l == tc.HGEMM_B_ROW_MAJOR else b)
    dc = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tc.hgemm_layout(a_l, b_l, da, M if a_l == tc.HGEMM_A_COL_MAJOR else K, db,
                    N if b_l == tc.HGEMM_B_ROW_MAJOR else K, dc, N, M, N, K)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, 255, 256, M - 1], rng.integers(0, M, 60)])
    cols = np.concatenate([[0, 63, 64, 127, 128, N - 1], rng.integers(0, N, 58)])
    rr, cc = np.meshgrid(rows, cols, indexing="ij")
    got = dc.cpu().numpy()[rr, cc]
    ref = oracle.entries(a, b, rr.ravel(), cc.ravel()).reshape(rr.shape)
    assert_close(got, ref, what=f"4096 {NAMES[layout]} sampled")

