"""Small cases on every kernel path, run by tests/test_debug_gpu.py in a
process that loads the -DHGEMM_DEBUG build (HGEMM_LIBRARY_VARIANT=debug):
each result must match the oracle within the tests' tolerance and leave no
device-side check or watchdog code behind. Exits non-zero on the first
failure, with a message."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402


def main() -> int:
    assert os.environ.get("HGEMM_LIBRARY_VARIANT") == "debug"
    from tensor_core_dense_fp16_gb300 import build
    build.build(debug=True)
    import torch
    import oracle
    import synth
    import tensor_core_dense_fp16_gb300 as tc
    from gpu_helpers import assert_close, oracle_threads, to_device

    tc.load()
    assert tc.hgemm_debug_build() == 1, "the debug variant was not loaded"
    assert tc.hgemm_debug_selftest() == 0

    def status(what):
        st = tc.hgemm_device_status()
        assert st == tc.HGEMM_OK, f"{what}: status {st}, check code {tc.hgemm_debug_code()}"

    # the product on every path, ragged shapes
    for path in (tc.HGEMM_PATH_TC, tc.HGEMM_PATH_TC_NARROW, tc.HGEMM_PATH_TC_PAIR, tc.HGEMM_PATH_TC_WIDE,
                 tc.HGEMM_PATH_SKINNY, tc.HGEMM_PATH_GENERIC):
        for M, N, K in [(300, 264, 200), (1000, 1000, 1000), (129, 8, 3000)]:
            a, b = synth.operands(M, N, K, seed=M + N + K, kind="uniform")
            da, db = to_device(a), to_device(b)
            dc = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            tc.hgemm_force_path(path)
            try:
                tc.hgemm(da, db, dc, M, N, K)
            finally:
                tc.hgemm_force_path(-1)
            status(f"path {path} {M}x{N}x{K}")
            assert_close(dc.cpu().numpy(), oracle.hgemm(a, b, nthreads=oracle_threads()),
                         what=f"debug build path {path} {M}x{N}x{K}")
    # fused epilogue and the other layouts (automatic paths)
    M, N, K = 600, 520, 400
    a, b = synth.operands(M, N, K, seed=5, kind="uniform")
    c0 = synth.operands(M, N, 1, seed=6, kind="uniform")[0][:, :1].repeat(N, axis=1)
    bias = synth.operands(1, N, 1, seed=7, kind="uniform")[1][:, 0].copy()
    da, db = to_device(a), to_device(b)
    dc = to_device(c0)
    tc.hgemm_ex(da, db, dc, M, N, K, 0.5, 1.0, to_device(bias), True)
    status("fused")
    assert_close(dc.cpu().numpy(), oracle.hgemm_ex(a, b, c0, 0.5, 1.0, bias, True, nthreads=oracle_threads()),
                 what="debug build fused")
    dat, dbt = to_device(np.ascontiguousarray(a.T)), to_device(np.ascontiguousarray(b.T))
    dc = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tc.hgemm_layout(tc.HGEMM_A_COL_MAJOR, tc.HGEMM_B_ROW_MAJOR, dat, M, dbt, N, dc, N, M, N, K, 1.0, 0.0,
                    None, False)
    status("layouts")
    assert_close(dc.cpu().numpy(), oracle.hgemm(a, b, nthreads=oracle_threads()), what="debug build layouts")
    # TRMM: tensor-core leaves (n a multiple of 64) and generic leaves
    for n, m in [(512, 100), (700, 64)]:
        rng = np.random.default_rng(n)
        a = rng.uniform(0, 1, size=(n, n)).astype(np.float16)
        b = rng.uniform(0, 1, size=(n, m)).astype(np.float16)
        dA, dB = to_device(np.ascontiguousarray(a.T)), to_device(np.ascontiguousarray(b.T))
        dC = torch.empty((m, n), dtype=torch.float16, device="cuda")
        tc.hgemm_trmm(dA, n, dB, n, dC, n, n, m, 1.0)
        status(f"trmm {n}x{m}")
        assert_close(dC.cpu().numpy().T, oracle.trmm(a, b, nthreads=oracle_threads()), what=f"debug trmm {n}")
    # TRSM, both orientations, with and without the workspace, and the fixed array
    n, m = 1000, 72
    a_col, b_col = synth.trsm_operands(n, m, 9)
    dA, dB = to_device(a_col), to_device(b_col)
    work = torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device="cuda")
    for op, ref in ((tc.HGEMM_OP_T, oracle.trsm(a_col.T, b_col.T, nthreads=oracle_threads())),
                    (tc.HGEMM_OP_N, oracle.trsm_n(a_col.T, b_col.T, nthreads=oracle_threads()))):
        for w in (None, work):
            dX = torch.empty((m, n), dtype=torch.float16, device="cuda")
            tc.hgemm_trsm_op(op, dA, n, dB, n, dX, n, n, m, 1.0, w)
            status(f"trsm op {op} ws {w is not None}")
            assert_close(dX.cpu().numpy().T, ref, what=f"debug trsm op {op} ws {w is not None}")
    dX = torch.empty((m, n), dtype=torch.float16, device="cuda")
    tc.hgemm_trsm_noalloc(dA, n, dB, n, dX, n, n, m, 1.0)
    status("trsm noalloc")
    print("debug build: every path clean")
    return 0


if __name__ == "__main__":
    sys.exit(main())
