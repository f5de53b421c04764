"""The triangular product of "异构计算中高性能TRMM与TRSM的递归算法实现" (§2.2,
B ← alpha·Aᵀ·B with A lower triangular, here out of place: C = alpha·Aᵀ·B)
through hgemm_trmm, against the oracle (GPU only).

Inputs follow the page's example (§5.1: rand(Float32) operands, uniform on
[0, 1)), here rounded to FP16. With nonnegative terms every intermediate
block the recursion rounds to FP16 is no larger than the final value, so the
per-element tolerance of the plain product applies."""

import numpy as np
import pytest

import oracle
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, oracle_threads, to_device, torch_cuda

pytestmark = pytest.mark.gpu


def trmm_inputs(n, m, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0, 1, size=(n, n)).astype(np.float16)
    b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
    return a, b


def run_trmm(a, b, alpha=1.0, pad=(0, 0, 0), poison_upper=False):
    """Column-major device buffers with pitches n + pad."""
    torch = torch_cuda()
    n, m = b.shape
    lda, ldb, ldc = n + pad[0], n + pad[1], n + pad[2]
    a_col = np.zeros((n, lda), np.float16)     # row c holds column c of A
    a_col[:, :n] = a.T
    if poison_upper:
        r, c = np.triu_indices(n, 1)            # A(r, c) with c > r: above the diagonal
        a_col[c, r] = np.nan
    b_col = np.zeros((m, ldb), np.float16)
    b_col[:, :n] = b.T
    c_col = np.full((m, ldc), 5.0, np.float16)
    da, db, dc = to_device(a_col), to_device(b_col), to_device(c_col)
    tc.hgemm_trmm(da, lda, db, ldb, dc, ldc, n, m, alpha)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    out = dc.cpu().numpy()
    assert np.all(out[:, n:] == 5.0), "pitch padding of C was written"
    return np.ascontiguousarray(out[:, :n].T)


@pytest.mark.parametrize("n,m", [(64, 32), (256, 100), (257, 64), (300, 136), (512, 256),
                                 (1000, 128), (4096, 256)])
def test_trmm_matches_oracle(n, m):
    a, b = trmm_inputs(n, m, seed=n + m)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b), ref, what=f"trmm {n}x{m}")


@pytest.mark.parametrize("n", [700, 1024])
def test_trmm_reads_only_the_lower_triangle(n):
    """NaN above the diagonal never reaches C: n = 700 takes the generic
    leaves (masked as they load), n = 1024 the tensor-core leaves (diagonal
    sub-blocks masked in shared memory, rows below them never loaded)."""
    m = 96
    a, b = trmm_inputs(n, m, seed=7)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b, poison_upper=True), ref, what=f"NaN above the diagonal, n={n}")


@pytest.mark.parametrize("n,m", [(64, 1), (192, 129), (320, 40), (448, 257), (576, 128)])
def test_trmm_tensor_core_leaf_orders(n, m):
    """n a multiple of 64: the leaves run on the tensor cores, with orders
    64, 192, 192 + 128, 256 + 192 and 320 + 256 split further (every leaf
    order a multiple of 64 up to 256), and ragged or single rows of B."""
    a, b = trmm_inputs(n, m, seed=31 + n)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b), ref, what=f"trmm {n}x{m}")


@pytest.mark.parametrize("n,m,slices", [(4096, 256, 4), (1280, 200, 4), (2048, 1100, 2), (1088, 1200, 2),
                                        (2048, 2500, 1)])
def test_trmm_leaves_split_over_clusters(n, m, slices):
    """With few leaf units (tiles of 128 rows of Bᵀ × leaves) every unit's K
    blocks are split over a cluster of four CTAs (four times the units fit on
    the GPU's 152 SMs at once) or two (twice do), the partial sums reduced
    through distributed shared memory; more units take the persistent kernel.
    Leaves of 256 columns carrying up to 3840 update columns (4096 x 256),
    leaves of other orders (1088) and ragged rows of B; n = 2048, m = 1100 has
    72 units, 1088 x 1200 has 60."""
    a, b = trmm_inputs(n, m, seed=53 + n + m)
    ref = oracle.trmm(a, b, alpha=0.75, nthreads=oracle_threads())
    assert_close(run_trmm(a, b, alpha=0.75), ref, what=f"trmm {n}x{m}, {slices} slices")


@pytest.mark.parametrize("path", [None, tc.HGEMM_PATH_GENERIC])
def test_trmm_leaf_kernels_agree(path):
    """The same product with the tensor-core leaves (default) and the generic
    leaves (forced): both within the tolerance, with a scale factor and
    pitches wider than the operands (multiples of 8, so TMA applies)."""
    n, m = 1280, 200
    a, b = trmm_inputs(n, m, seed=41)
    ref = oracle.trmm(a, b, alpha=0.25, nthreads=oracle_threads())
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        out = run_trmm(a, b, alpha=0.25, pad=(8, 8, 16))
    finally:
        if path is not None:
            tc.hgemm_force_path(-1)
    assert_close(out, ref, what=f"trmm 1280x200, path {path}")


@pytest.mark.parametrize("pad", [(8, 16, 8), (3, 5, 1)])
def test_trmm_pitches_and_alpha(pad):
    """Wider pitches (multiples of 8: tensor-core updates; odd ones: the
    generic loader) and a scale factor."""
    n, m = 600, 72
    a, b = trmm_inputs(n, m, seed=11 + pad[0])
    ref = oracle.trmm(a, b, alpha=0.5, nthreads=oracle_threads())
    assert_close(run_trmm(a, b, alpha=0.5, pad=pad), ref, what=f"trmm pad {pad}")


def test_trmm_repeatable():
    torch = torch_cuda()
    n, m = 1024, 64
    a, b = trmm_inputs(n, m, seed=3)
    first = run_trmm(a, b)
    for _ in range(3):
        assert np.array_equal(run_trmm(a, b).view(np.uint16), first.view(np.uint16))


@pytest.mark.parametrize("path", [None, tc.HGEMM_PATH_TC_PAIR, tc.HGEMM_PATH_TC, tc.HGEMM_PATH_TC_NARROW,
                                  tc.HGEMM_PATH_GENERIC])
def test_trmm_equal_levels(path):
    """n = 2048: each level of the recursion holds equal updates at a constant
    stride (2 of 1024 columns, then 4 of 512, 8 of 256 ...). On the pair path
    (chosen, or forced) a level runs as one batched launch; another forced
    path runs it update by update. m = 300 leaves a ragged row of tiles,
    with a scale factor and pitches wider than the operands."""
    n, m = 2048, 300
    a, b = trmm_inputs(n, m, seed=21)
    ref = oracle.trmm(a, b, alpha=0.5, nthreads=oracle_threads())
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        out = run_trmm(a, b, alpha=0.5, pad=(8, 16, 24))
    finally:
        if path is not None:
            tc.hgemm_force_path(-1)
    assert_close(out, ref, what=f"trmm 2048x300, path {path}")


def test_trmm_equal_levels_wide_m():
    """n = 1024, m = 1000: the batched levels with several tile rows of C per
    update and a ragged last row."""
    n, m = 1024, 1000
    a, b = trmm_inputs(n, m, seed=23)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b), ref, what="trmm 1024x1000")


def test_trmm_carried_and_separate_updates():
    """n = 2048, m = 8200 (automatic path): the updates of the 1024-blocks
    and below are carried by the leaves, the top one (8200 × 1024 × 1024
    multiply-adds, above 2^33) runs as a product of its own after them."""
    n, m = 2048, 8200
    a, b = trmm_inputs(n, m, seed=29)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b), ref, what="trmm 2048x8200")


# ---- signed operands: the envelope of the recursion's FP16 intermediates

def signed_inputs(n, m, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(-1, 1, size=(n, n)).astype(np.float16)
    b = rng.uniform(-1, 1, size=(n, m)).astype(np.float16)
    return a, b


def separate_update_levels(n, m, tc_leaves, forced=False):
    """Levels of the recursion whose updates run as products of their own
    (each rounds the rows it updates to FP16 once more); the other updates
    are carried by the tensor-core leaves, inside their single rounding.
    Blocks split at half rounded up to 64 and stop at 256; a leaf carries an
    update of at most 2^33 multiply-adds."""
    levels = set()

    def walk(s, depth):
        if s <= 256:
            return
        s1 = ((s // 2 + 63) // 64) * 64
        if not tc_leaves or forced or m * s1 * (s - s1) > 2 ** 33:
            levels.add(depth)
        walk(s1, depth + 1)
        walk(s - s1, depth + 1)

    walk(n, 0)
    return len(levels)


@pytest.mark.parametrize("n,m", [(2048, 512), (4096, 256), (8192, 512)])
def test_trmm_signed_single_rounding(n, m):
    """Operands uniform on [-1, 1]: where every update is carried by the
    tensor-core leaves (n a multiple of 64, m·s1·s2 <= 2^33 for every
    update, including n = 8192 with m = 512), each output is one FP32 sum
    rounded once, like a product, and the product's tolerance holds."""
    assert separate_update_levels(n, m, tc_leaves=True) == 0
    a, b = signed_inputs(n, m, seed=101 + n)
    ref = oracle.trmm(a, b, nthreads=oracle_threads())
    assert_close(run_trmm(a, b), ref, what=f"signed trmm {n}x{m}")


@pytest.mark.parametrize("n,m,path", [(2048, 8200, None), (1000, 128, None),
                                      (2048, 300, tc.HGEMM_PATH_TC_PAIR)])
def test_trmm_signed_separate_updates_envelope(n, m, path):
    """Operands uniform on [-1, 1] where some updates run as separate
    products (a large update, generic leaves at n = 1000, or a forced path):
    each such level rounds a partial sum P of the output to FP16 once more,
    an error of at most 2^-11·|P| <= 2^-11·S with S = sum |A(k,i)|·|B(k,j)|
    (the oracle's product of the absolute values). With R such levels the
    product's tolerance widens by R·2^-11·S; with nonnegative operands
    S = |C| and the widening is inside the product's tolerance, which the
    other tests apply. A dropped or doubled update, or a wrong sign, is off
    by far more than the widening."""
    a, b = signed_inputs(n, m, seed=211 + n + m)
    r = separate_update_levels(n, m, tc_leaves=(n % 64 == 0), forced=path is not None)
    assert r >= 1
    ref = oracle.trmm(a, b, nthreads=oracle_threads()).astype(np.float64)
    s_abs = oracle.trmm(np.abs(a), np.abs(b), nthreads=oracle_threads()).astype(np.float64)
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        got = run_trmm(a, b).astype(np.float64)
    finally:
        if path is not None:
            tc.hgemm_force_path(-1)
    assert not np.isnan(got).any()
    err = np.abs(got - ref)
    lim = 1e-2 * np.maximum(1.0, np.abs(ref)) + r * 2.0 ** -11 * s_abs * (1 + 2.0 ** -10)
    assert np.all(err <= lim), (
        f"signed trmm {n}x{m} ({r} separate levels): {int((err > lim).sum())} outputs out of "
        f"the envelope, worst {float((err / lim).max()):.3g}x")
    # a dropped update of the top level would leave rows [0, s1) off by the
    # whole update, far outside the envelope there
    s1 = ((n // 2 + 63) // 64) * 64
    upd = (a[s1:, :s1].astype(np.float64).T @ b[s1:].astype(np.float64))
    assert np.mean(np.abs(upd) > lim[:s1]) > 0.5
