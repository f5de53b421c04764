"""Multi-process host logic of the benchmark's replica mode, on CPU with gloo
(world size 2): the slowest rank's time and the whole-job throughput."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.0][rank]
        slowest = bench.reduce_max(local_ms, dist, "cpu")
        value = bench.whole_job_tflops(world, 10, 2.0e12, slowest)
        out[rank] = (slowest, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == 55.0
        # 2 ranks x 10 steps x 2e12 flops over 55 ms
        assert value == pytest.approx(2 * 10 * 2.0e12 / 0.055 / 1e12)


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(12.5, None, "cpu") == 12.5
    assert bench.whole_job_tflops(1, 4, 1.0e12, 2.0) == pytest.approx(2000.0)


def test_reference_arm_under_two_ranks():
    """`bench.py --impl reference` launched as two ranks (torchrun, as for an
    N-GPU run): rank 0 alone times the oracle and prints the one line, the
    other rank exits 0 without work."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl",
           "reference", "--workload", "hgemm_256", "--steps", "1", "--warmup", "1", "--gpus", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
