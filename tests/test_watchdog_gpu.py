"""Failure detection without a GPU fault: every wait inside the kernels is
bounded in time. The testing hook makes a kernel's TMA producer withhold one
barrier arrival (its copies still land), so the MMA issuer's wait runs out;
the kernel must record the timeout, drain, free TMEM and return, the host
must read HGEMM_ERR_TIMEOUT, and the context must stay usable."""

import numpy as np
import pytest

import oracle
import synth
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, run_gpu, to_device, torch_cuda


def test_hook_arguments_are_checked():
    tc.load()
    with pytest.raises(tc.HgemmError):
        tc.hgemm_debug_inject(99)
    tc.hgemm_debug_inject(tc.HGEMM_INJECT_NONE)
    tc.hgemm_set_wait_timeout(0)


@pytest.mark.gpu
@pytest.mark.parametrize("path", [tc.HGEMM_PATH_TC, tc.HGEMM_PATH_TC_NARROW, tc.HGEMM_PATH_TC_PAIR,
                                  tc.HGEMM_PATH_TC_WIDE,
                                  tc.HGEMM_PATH_SKINNY])
def test_withheld_arrival_times_out_and_the_context_survives(path):
    torch = torch_cuda()
    M = N = K = 512
    a, b = synth.operands(M, N, K, seed=31, kind="uniform")
    da, db = to_device(a), to_device(b)
    dc = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    tc.hgemm_set_wait_timeout(50_000_000)   # 50 ms per wait
    tc.hgemm_debug_inject(tc.HGEMM_INJECT_DROP_ARRIVAL)
    tc.hgemm_force_path(path)
    try:
        tc.hgemm(da, db, dc, M, N, K)
        assert tc.hgemm_device_status() == tc.HGEMM_ERR_TIMEOUT
        # the word was cleared by the read
        assert tc.hgemm_device_status() == tc.HGEMM_OK
    finally:
        tc.hgemm_debug_inject(tc.HGEMM_INJECT_NONE)
        tc.hgemm_set_wait_timeout(0)
        tc.hgemm_force_path(-1)
    # the same context computes correctly afterwards
    ref = oracle.hgemm(a, b)
    assert_close(run_gpu(a, b, path=path), ref, what=f"after timeout, path {path}")


@pytest.mark.gpu
@pytest.mark.parametrize("m", [256, 8192], ids=["split-clusters", "persistent"])
def test_withheld_arrival_in_the_trmm_leaf_kernel(m):
    """The same on the triangular product: the tensor-core leaf kernel (the
    first launch of hgemm_trmm, n a multiple of 64) records the timeout and
    returns; afterwards the same context computes the product correctly.
    m = 256: 4 leaf units, each split over a cluster of four CTAs (the CTAs
    without K blocks still wait for partials that never come); m = 8192: 128
    units on the persistent kernel."""
    torch = torch_cuda()
    n = 512
    rng = np.random.default_rng(37)
    a = rng.uniform(0, 1, size=(n, n)).astype(np.float16)
    b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
    da, db = to_device(np.ascontiguousarray(a.T)), to_device(np.ascontiguousarray(b.T))
    dc = torch.zeros((m, n), dtype=torch.float16, device="cuda")
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    tc.hgemm_set_wait_timeout(50_000_000)   # 50 ms per wait
    tc.hgemm_debug_inject(tc.HGEMM_INJECT_DROP_ARRIVAL)
    try:
        tc.hgemm_trmm(da, n, db, n, dc, n, n, m, 1.0)
        assert tc.hgemm_device_status() == tc.HGEMM_ERR_TIMEOUT
        assert tc.hgemm_device_status() == tc.HGEMM_OK
    finally:
        tc.hgemm_debug_inject(tc.HGEMM_INJECT_NONE)
        tc.hgemm_set_wait_timeout(0)
    tc.hgemm_trmm(da, n, db, n, dc, n, n, m, 1.0)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    ref = oracle.trmm(a, b)
    assert_close(np.ascontiguousarray(dc.cpu().numpy().T), ref, what="trmm after timeout")


@pytest.mark.gpu
def test_withheld_arrival_in_the_one_launch_solve():
    """The persistent TRSM launch (hgemm_trsm_ws, chain schedule): every
    CTA's producer withholds its first arrival, so the MMA issuers' waits run
    out; each CTA raises its abort flag, the launch's abort word reaches the
    CTAs waiting at the grid barrier, and all drain, free TMEM and return.
    Afterwards the same context solves correctly."""
    torch = torch_cuda()
    n, m = 1024, 64
    a_col, b_col = synth.trsm_operands(n, m, 43)
    da, db = to_device(a_col), to_device(b_col)
    dx = torch.zeros((m, n), dtype=torch.float16, device="cuda")
    work = torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device="cuda")
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    tc.hgemm_set_wait_timeout(50_000_000)   # 50 ms per wait
    tc.hgemm_debug_inject(tc.HGEMM_INJECT_DROP_ARRIVAL)
    tc.hgemm_force_trsm_schedule(tc.HGEMM_TRSM_CHAIN)
    try:
        tc.hgemm_trsm_ws(da, n, db, n, dx, n, n, m, 1.0, work)
        assert tc.hgemm_trsm_last_schedule() in (tc.HGEMM_TRSM_CHAIN_FUSED, tc.HGEMM_TRSM_CHAIN_SPLIT)
        assert tc.hgemm_device_status() == tc.HGEMM_ERR_TIMEOUT
        assert tc.hgemm_device_status() == tc.HGEMM_OK
    finally:
        tc.hgemm_debug_inject(tc.HGEMM_INJECT_NONE)
        tc.hgemm_set_wait_timeout(0)
        tc.hgemm_force_trsm_schedule(tc.HGEMM_TRSM_AUTO)
    tc.hgemm_trsm_ws(da, n, db, n, dx, n, n, m, 1.0, work)
    assert tc.hgemm_trsm_last_schedule() in (tc.HGEMM_TRSM_CHAIN_FUSED, tc.HGEMM_TRSM_CHAIN_SPLIT)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    ref = oracle.trsm(a_col.T, b_col.T)
    assert_close(np.ascontiguousarray(dx.cpu().numpy().T), ref, what="trsm after a timeout")
