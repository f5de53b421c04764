"""hgemm_trsm_noalloc: the triangular solve for callers that cannot allocate
device memory (their memory all belongs to another allocator, or they must
not pay cudaMalloc's synchronisation). Its workspace is a fixed 8 MiB array
inside the library instead of one the caller passes in.

Checked through the C ABI against the entry point that takes a caller-owned
workspace (hgemm_trsm_ws, same algorithm) and against hgemm_trsm, within the
TRSM tests' tolerance, on two calls in a row: the second, smaller solve
reuses the array the first one filled, so a stale entry it read would show.
This file is collected last (GPU only)."""

import numpy as np
import pytest

import synth
import tensor_core_dense_fp16_gb300 as tc
from gpu_helpers import assert_close, to_device, torch_cuda

pytestmark = pytest.mark.gpu


def _solve(entry, a_col, b_col, n, m):
    """X for Aᵀ·X = B (column-major device buffers, pitches n) through one entry point."""
    torch = torch_cuda()
    da, db = to_device(a_col), to_device(b_col)
    dx = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
    if entry == "noalloc":
        tc.hgemm_trsm_noalloc(da, n, db, n, dx, n, n, m, 1.0)
    elif entry == "ws":
        work = torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device="cuda")
        tc.hgemm_trsm_ws(da, n, db, n, dx, n, n, m, 1.0, work)
    else:
        tc.hgemm_trsm(da, n, db, n, dx, n, n, m, 1.0)
    assert tc.hgemm_device_status() == tc.HGEMM_OK
    torch.cuda.synchronize()
    return np.ascontiguousarray(dx.cpu().numpy().T)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    tc.load()
    for n, m, seed in [(2048, 512, 71), (1000, 300, 72)]:  # 4 diagonal blocks, then 2 (one of order 488)
        a_col, b_col = synth.trsm_operands(n, m, seed)
        got = _solve("noalloc", a_col, b_col, n, m)
        assert_close(got, _solve("ws", a_col, b_col, n, m), what=f"noalloc vs ws {n}x{m}")
        assert_close(got, _solve("plain", a_col, b_col, n, m), what=f"noalloc vs trsm {n}x{m}")


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
