"""The fused product hgemm_ex, C = f(alpha·A·B + beta·C + bias[j]) with
f = ReLU or the identity ("GPU架构与CUDA", 核函数融合), against the oracle's
fused variant on every path (GPU only)."""

import numpy as np
import pytest

import oracle
import synth
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, oracle_threads, to_device, torch_cuda

pytestmark = pytest.mark.gpu

PATHS = [None, tc.HGEMM_PATH_TC, tc.HGEMM_PATH_TC_NARROW, tc.HGEMM_PATH_TC_PAIR, tc.HGEMM_PATH_TC_WIDE,
         tc.HGEMM_PATH_SKINNY, tc.HGEMM_PATH_GENERIC]
EPILOGUES = [  # alpha, beta, with bias, relu
    (1.0, 0.0, True, True),      # the page's matmul + bias + ReLU
    (1.0, 1.0, False, False),    # accumulate into C (a TRMM off-diagonal update)
    (-1.25, -0.5, True, True),
    (0.5, 2.0, True, False),
]


def run_ex(a, b, c_old, alpha, beta, bias, relu, path=None, split=None):
    torch = torch_cuda()
    M, K = a.shape
    N = b.shape[0]
    da, db = to_device(a), to_device(b)
    dc = to_device(c_old) if c_old is not None else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                                device="cuda")
    dbias = to_device(bias) if bias is not None else None
    if path is not None:
        tc.hgemm_force_path(path)
    if split is not None:
        tc.hgemm_force_split(*split)
    try:
        tc.hgemm_ex(da, db, dc, M, N, K, alpha, beta, dbias, relu)
    finally:
        tc.hgemm_force_path(-1)
        tc.hgemm_force_split(0, 0)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    return dc.cpu().numpy()


def inputs(M, N, K, seed):
    a, b = synth.operands(M, N, K, seed=seed, kind="uniform")
    rng = np.random.default_rng(seed)
    c_old = rng.uniform(-4, 4, size=(M, N)).astype(np.float16)
    bias = rng.uniform(-2, 2, size=N).astype(np.float16)
    return a, b, c_old, bias


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("alpha,beta,with_bias,relu", EPILOGUES)
def test_fused_matches_oracle(path, alpha, beta, with_bias, relu):
    M, N, K = 1000, 520, 384   # ragged in M and N against every tile shape
    a, b, c_old, bias = inputs(M, N, K, seed=4242)
    bias = bias if with_bias else None
    ref = oracle.hgemm_ex(a, b, c_old, alpha, beta, bias, relu, nthreads=oracle_threads())
    got = run_ex(a, b, c_old, alpha, beta, bias, relu, path=path)
    assert_close(got, ref, what=f"path {path} alpha {alpha} beta {beta} bias {with_bias} relu {relu}")


@pytest.mark.parametrize("split", [(2, 128), (2, 256), (3, 256), (4, 256)])
def test_fused_split_k_configurations(split):
    M, N, K = 256 * 9 - 13, 248, 64 * 9 + 24
    a, b, c_old, bias = inputs(M, N, K, seed=99 + split[0])
    ref = oracle.hgemm_ex(a, b, c_old, 0.75, 1.0, bias, True, nthreads=oracle_threads())
    got = run_ex(a, b, c_old, 0.75, 1.0, bias, True, path=tc.HGEMM_PATH_SKINNY, split=split)
    assert_close(got, ref, what=f"split {split}")


@pytest.mark.parametrize("path", PATHS)
def test_fused_integer_operands_bit_exact(path):
    """Integer A, B, C_old and bias, power-of-two alpha and beta: every FP32
    step is exact, so the result must equal the oracle bit for bit."""
    rng = np.random.default_rng(7)
    M, N, K = 300, 136, 256
    a = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    b = rng.integers(-2, 3, size=(N, K)).astype(np.float16)
    c_old = rng.integers(-100, 101, size=(M, N)).astype(np.float16)
    bias = rng.integers(-30, 31, size=N).astype(np.float16)
    ref = oracle.hgemm_ex(a, b, c_old, 2.0, -1.0, bias, True)
    got = run_ex(a, b, c_old, 2.0, -1.0, bias, True, path=path)
    assert_close(got, ref, exact=True, what=f"integer fused, path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_fused_beta_zero_does_not_read_c(path):
    M, N, K = 200, 136, 72
    a, b, _, bias = inputs(M, N, K, seed=3)
    nan_c = np.full((M, N), np.nan, np.float16)
    got = run_ex(a, b, nan_c, 1.5, 0.0, bias, False, path=path)
    assert not np.isnan(got.astype(np.float32)).any()
    assert_close(got, oracle.hgemm_ex(a, b, None, 1.5, 0.0, bias, False), what=f"beta 0, path {path}")


def test_fused_identity_epilogue_is_the_plain_product():
    torch = torch_cuda()
    a, b, spec = synth.workload("hgemm_2048")
    M, N, K = spec["M"], spec["N"], spec["K"]
    da, db = to_device(a), to_device(b)
    c1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    c2 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tc.hgemm(da, db, c1, M, N, K)
    tc.hgemm_ex(da, db, c2, M, N, K, 1.0, 0.0, None, False)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("beta,with_bias,relu", [(0.0, False, False), (1.0, True, True), (-2.0, False, True)])
def test_fused_empty_sum(beta, with_bias, relu):
    """K = 0: C := f(beta·C_old + bias)."""
    M, N = 77, 40
    rng = np.random.default_rng(11)
    c_old = rng.uniform(-3, 3, size=(M, N)).astype(np.float16)
    bias = rng.uniform(-1, 1, size=N).astype(np.float16) if with_bias else None
    a = np.zeros((M, 0), np.float16)
    b = np.zeros((N, 0), np.float16)
    torch = torch_cuda()
    da = torch.empty((M, 8), dtype=torch.float16, device="cuda")   # any valid pointers
    db = torch.empty((N, 8), dtype=torch.float16, device="cuda")
    dc = to_device(c_old)
    dbias = to_device(bias) if bias is not None else None
    tc.hgemm_ex(da, db, dc, M, N, 0, 1.0, beta, dbias, relu)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    ref = oracle.hgemm_ex(a, b, c_old, 1.0, beta, bias, relu)
    assert_close(dc.cpu().numpy(), ref, exact=True, what="K = 0")


def test_fused_8192_cube_sampled():
    """The headline shape with the accumulate-plus-bias-plus-ReLU epilogue,
    checked on sampled entries."""
    torch = torch_cuda()
    a, b, spec = synth.workload("hgemm_8192")
    M, N, K = spec["M"], spec["N"], spec["K"]
    rng = np.random.default_rng(8)
    c_old = rng.standard_normal((M, N), dtype=np.float32).astype(np.float16)
    bias = rng.uniform(-1, 1, size=N).astype(np.float16)
    da, db, dc, dbias = to_device(a), to_device(b), to_device(c_old), to_device(bias)
    tc.hgemm_ex(da, db, dc, M, N, K, 1.0, 1.0, dbias, True)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    got = dc.cpu().numpy()
    rows = np.concatenate([rng.integers(0, M, 2000), [0, 255, 256, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 2000), [0, 511, 512, N - 1]])
    ref = oracle.entries_ex(a, b, rows, cols, c_old, 1.0, 1.0, bias, True)
    assert_close(got[rows, cols], ref, what="8192 fused sampled")


@pytest.mark.parametrize("path", PATHS)
def test_fused_guard_bands_untouched(path):
    torch = torch_cuda()
    M, N, K = 200, 136, 72
    a, b, c_old, bias = inputs(M, N, K, seed=21)
    ref = oracle.hgemm_ex(a, b, c_old, 1.0, 1.0, bias, True)
    sentinel = 0x7E01
    pad = 4096
    buf = torch.full((pad + M * N + pad,), sentinel, dtype=torch.int16, device="cuda")
    buf[pad:pad + M * N] = torch.from_numpy(c_old.view(np.int16).reshape(-1)).to("cuda")
    da, db, dbias = to_device(a), to_device(b), to_device(bias)
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        assert tc.load().hgemm_ex(da.data_ptr(), db.data_ptr(), buf.data_ptr() + 2 * pad, M, N, K, 1.0, 1.0,
                                  dbias.data_ptr(), 1, torch.cuda.current_stream().cuda_stream) == 0
    finally:
        tc.hgemm_force_path(-1)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    host = buf.cpu().numpy()
    assert np.all(host[:pad] == sentinel) and np.all(host[pad + M * N:] == sentinel)
    assert_close(host[pad:pad + M * N].view(np.float16).reshape(M, N), ref, what=f"guarded fused {path}")


# ---------------------------------------------------------------------------
# hgemm_strided: sub-matrices with row pitches


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("pitch_pad", [0, 8, 5])
def test_strided_sub_matrices(path, pitch_pad):
    """Operands and C inside larger arrays (pitches wider than the rows, by 8
    elements or by 5, which sends every path to the generic loader); the
    padding around C must be left untouched."""
    torch = torch_cuda()
    M, N, K = 300, 200, 136
    lda, ldb, ldc = K + pitch_pad, K + pitch_pad + 8, N + pitch_pad
    a, b, c_old, bias = inputs(M, N, K, seed=600 + pitch_pad)
    big_a = np.zeros((M, lda), np.float16); big_a[:, :K] = a
    big_b = np.zeros((N, ldb), np.float16); big_b[:, :K] = b
    big_c = np.full((M, ldc), 7.0, np.float16); big_c[:, :N] = c_old
    da, db, dc, dbias = to_device(big_a), to_device(big_b), to_device(big_c), to_device(bias)
    ref = oracle.hgemm_ex(a, b, c_old, 0.5, 1.0, bias, True)
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        tc.hgemm_strided(da, lda, db, ldb, dc, ldc, M, N, K, 0.5, 1.0, dbias, True)
    finally:
        tc.hgemm_force_path(-1)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    got = dc.cpu().numpy()
    assert_close(got[:, :N], ref, what=f"strided path {path} pad {pitch_pad}")
    assert np.all(got[:, N:] == 7.0)


def test_strided_offset_blocks_of_one_matrix():
    """A, B and C as blocks of larger column-major matrices, as the TRMM
    recursion uses them (offsets into the same arrays, pitch n)."""
    torch = torch_cuda()
    n, m = 512, 256
    rng = np.random.default_rng(9)
    big_a = rng.uniform(-1, 1, size=(n, n)).astype(np.float16)   # rows: pitch n
    big_b = rng.uniform(-1, 1, size=(n, n)).astype(np.float16)
    big_c = np.zeros((n, n), np.float16)
    da, db, dc = to_device(big_a), to_device(big_b), to_device(big_c)
    h = n // 2
    # C[h:, :m] = A[h:, h:] · B-block whose column j is big_b[j, h:]
    tc.hgemm_strided(da.data_ptr() + 2 * (h * n + h), n, db.data_ptr() + 2 * h, n,
                     dc.data_ptr() + 2 * (h * n), n, h, m, h)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    got = dc.cpu().numpy()
    ref = oracle.hgemm(big_a[h:, h:], big_b[:m, h:])
    assert_close(got[h:, :m], ref, what="offset blocks")
    assert np.all(got[:h] == 0) and np.all(got[h:, m:] == 0)
