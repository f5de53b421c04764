"""hgemm_trsm_noalloc: the triangular solve for callers that cannot allocate
device memory (their memory all belongs to another allocator, or they must
not pay cudaMalloc's synchronisation). Its workspace is a fixed 8 MiB array
inside the library instead of one the caller passes in.

Checked through the C ABI on two calls in a row (the second, smaller solve
reuses the array the first one filled, so a stale entry it read would show):
against the oracle directly, and against the entry point that takes a
caller-owned workspace (hgemm_trsm_ws, same algorithm) and hgemm_trsm, within
the TRSM tests' tolerance. The calls must leave the device's free memory
unchanged. This file is collected last (GPU only)."""

import numpy as np
import pytest

import oracle
import synth
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, oracle_threads, torch_cuda

pytestmark = pytest.mark.gpu

CASES = [(2048, 512, 71), (1000, 300, 72)]  # 4 diagonal blocks, then 2 (one of order 488)


def _buffers(n, m, seed):
    """Device operands (column-major, pitches n) and a NaN-filled X for one case."""
    torch = torch_cuda()
    a_col, b_col = synth.trsm_operands(n, m, seed)
    da = torch.from_numpy(a_col).to("cuda")
    db = torch.from_numpy(b_col).to("cuda")
    dx = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
    return a_col, b_col, da, db, dx


def _noalloc(da, db, dx, n, m):
    dx.fill_(float("nan"))
    tc.hgemm_trsm_noalloc(da, n, db, n, dx, n, n, m, 1.0)


def _result(dx):
    torch = torch_cuda()
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    return np.ascontiguousarray(dx.cpu().numpy().T)


def test_noalloc_matches_the_oracle_and_the_workspace_entry_point_on_two_calls():
    torch = torch_cuda()
    tc.load()
    bufs = [_buffers(n, m, seed) for n, m, seed in CASES]
    # one call of each shape first, so that every kernel the solves use is
    # loaded before free memory is read (lazy module loading takes device memory)
    for (n, m, _), (_, _, da, db, dx) in zip(CASES, bufs):
        _noalloc(da, db, dx, n, m)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    got = []
    for (n, m, _), (_, _, da, db, dx) in zip(CASES, bufs):
        _noalloc(da, db, dx, n, m)
        got.append(_result(dx))
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, f"device free memory changed by {free_before - free_after} bytes"

    for (n, m, _), (a_col, b_col, da, db, _), x in zip(CASES, bufs, got):
        ref = oracle.trsm(a_col.T, b_col.T, nthreads=oracle_threads())
        assert_close(x, ref, what=f"noalloc vs oracle {n}x{m}")
        work = torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device="cuda")
        dx_ws = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        tc.hgemm_trsm_ws(da, n, db, n, dx_ws, n, n, m, 1.0, work)
        assert_close(x, _result(dx_ws), what=f"noalloc vs ws {n}x{m}")
        dx_plain = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        tc.hgemm_trsm(da, n, db, n, dx_plain, n, n, m, 1.0)
        assert_close(x, _result(dx_plain), what=f"noalloc vs trsm {n}x{m}")


def test_noalloc_rejects_triangles_beyond_its_array():
    torch = torch_cuda()
    tc.load()
    assert tc.hgemm_trsm_workspace_size(8192) <= tc.HGEMM_TRSM_NOALLOC_MAX_BYTES
    assert tc.hgemm_trsm_workspace_size(8193) > tc.HGEMM_TRSM_NOALLOC_MAX_BYTES
    n, m = 8193, 1
    da = torch.zeros((n, n), dtype=torch.float16, device="cuda")
    db = torch.zeros((m, n), dtype=torch.float16, device="cuda")
    with pytest.raises(tc.HgemmError) as err:
        tc.hgemm_trsm_noalloc(da, n, db, n, db, n, n, m, 1.0)
    assert err.value.status == tc.HGEMM_ERR_INVALID_ARG
