"""Shared helpers of the GPU tests: upload, call through the C ABI, compare."""

from __future__ import annotations

import os

import numpy as np

import oracle
import tensor_core_dense_fp16_gb300 as tc

# Acceptance per element for random inputs: |gpu - ref| <= TOL * max(1, |ref|),
# with ref the FP64-accumulated oracle rounded once to FP16.
TOL = 1e-2


def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def library():
    """The built library; GPU tests fail (not skip) when it is missing."""
    return tc.load()


def to_device(x: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda")


def run_gpu(a: np.ndarray, b: np.ndarray, path: int | None = None, stream=None) -> np.ndarray:
    """C = A·B through hgemm on the GPU; a is (M, K), b is (N, K)."""
    torch = torch_cuda()
    library()
    M, K = a.shape
    N = b.shape[0]
    da, db = to_device(a), to_device(b)
    dc = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    if path is not None:
        tc.hgemm_force_path(path)
    try:
        tc.hgemm(da, db, dc, M, N, K, stream)
    finally:
        if path is not None:
            tc.hgemm_force_path(-1)
    assert tc.hgemm_device_status(stream) == tc.HGEMM_OK
    torch.cuda.synchronize()
    return dc.cpu().numpy()


def oracle_threads() -> int:
    return os.cpu_count() or 1


def assert_close(got: np.ndarray, ref: np.ndarray, exact: bool = False, what: str = ""):
    """Per-element check against the oracle. exact: equal values (+0 == -0)."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    assert not np.isnan(g).any(), f"{what}: NaN in GPU output"
    if exact:
        bad = np.nonzero(g != r)
        assert bad[0].size == 0, (
            f"{what}: {bad[0].size} mismatches, first at {tuple(int(v[0]) for v in bad)}: "
            f"gpu {g[bad][0]} oracle {r[bad][0]}")
        return
    err = np.abs(g - r)
    lim = TOL * np.maximum(1.0, np.abs(r))
    bad = np.nonzero(err > lim)
    assert bad[0].size == 0, (
        f"{what}: {bad[0].size} elements out of tolerance, worst "
        f"{float((err / lim).max()):.3g}x the bound at "
        f"{tuple(int(v[np.argmax((err / lim)[bad])]) for v in bad)}")
