#!/usr/bin/env python
"""Benchmark of the FP16 HGEMM C = A·B on GB300.

One step is one C = A·B through the C ABI on the workload's operands, which
are resident in HBM before the timed region starts. Every timed launch is
bracketed by CUDA events on the stream it is launched on, and L2 is flushed
(a write of twice its size) before each launch, outside the events.

Prints one JSON line on rank 0. `value` is the work of one step on every
rank over the median step time (the slowest rank's median under torchrun,
where each rank runs an independent replica of the workload on its own GPU:
the product does not shard, there is no data-path collective). In the
default run the line also carries `configs`: the other configurations of the
problem (256-cube uniform and integer, 2048-cube, ragged 1000-cube, skinny
4096×256×4096) timed the same way after the headline, each with its median,
TFLOP/s and roofline fraction. `clocks` comes from in-process NVML samples
(about every millisecond) taken inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

`--impl reference` times the oracle (plain C, FP64) on this host's cores on a
bounded sample of the same workload: the comparison program, not a target.
"""

from __future__ import annotations

import argparse
import datetime
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "HGEMM TFLOP/s (2MNK/t) at 8192³ fp16 and % of GB300 dense FP16 peak"


def metric_for(name, spec):
    """The headline metric for the 8192-cube; the same quantity named by shape
    for the other workloads."""
    if name == DEFAULT_WORKLOAD:
        return METRIC
    if spec.get("op") == "trmm":
        return f"TRMM TFLOP/s (n(n+1)m/t) at n={spec['n']}, m={spec['m']} fp16"
    if spec.get("op") == "trsm":
        return f"TRSM TFLOP/s (n^2 m/t) at n={spec['n']}, m={spec['m']} fp16"
    if spec.get("op") == "trsm_n":
        return f"TRSM (A X = B) TFLOP/s (n^2 m/t) at n={spec['n']}, m={spec['m']} fp16"
    return f"HGEMM TFLOP/s (2MNK/t) at {spec['M']}x{spec['N']}x{spec['K']} fp16"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "hgemm_8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense FP16 : BF16 tensor throughput on this architecture (both
# 2.25 PFLOP/s dense per GPU), so the BF16 measured peak is the FP16 peak.
FP16_PER_BF16 = 1.0
DESCRIPTIONS = {
    "hgemm_8192": "M=N=K=8192 fp16; A row-major N(0,1), B col-major N(0,1)/sqrt(K); "
                  "fp32 accumulate; C fp16 row-major",
    "hgemm_2048": "M=N=K=2048 fp16; A, B uniform[-1,1]",
    "hgemm_1000_ragged": "M=N=K=1000 fp16 (ragged tiles); A, B uniform[-1,1]",
    "hgemm_256": "M=N=K=256 fp16; A, B uniform[-1,1]",
    "hgemm_256_int": "M=N=K=256 fp16; A, B integers in {-2..2}",
    "hgemm_4096x256x4096_skinny": "M=4096, N=256, K=4096 fp16; A, B uniform[-1,1] "
                                  "(bandwidth-bound)",
    "trmm_8192": "C = A^T B, A 8192x8192 lower triangular, B 8192x8192, column-major fp16; "
                 "A, B uniform[0,1]",
    "trmm_4096x256": "C = A^T B, A 4096x4096 lower triangular, B 4096x256, column-major fp16; "
                     "A, B uniform[0,1]",
    "trsm_8192": "solve A^T X = B, A 8192x8192 lower triangular (diagonal uniform[1,2], "
                 "below it uniform[0,1/n]), B 8192x8192 uniform[0,1], column-major fp16",
    "trsm_4096x256": "solve A^T X = B, A 4096x4096 lower triangular (diagonal uniform[1,2], "
                     "below it uniform[0,1/n]), B 4096x256 uniform[0,1], column-major fp16",
    "trsm_n_8192": "solve A X = B, A 8192x8192 lower triangular (diagonal uniform[1,2], "
                   "below it uniform[0,1/n]), B 8192x8192 uniform[0,1], column-major fp16",
    "trsm_n_4096x256": "solve A X = B, A 4096x4096 lower triangular (diagonal uniform[1,2], "
                       "below it uniform[0,1/n]), B 4096x256 uniform[0,1], column-major fp16",
}


def trmm_launches(n, m, leaf=256):
    """Kernel launches of one hgemm_trmm (pitches n, aligned operands): the
    batched leaves, then per recursion level either one batched launch (two or
    more equal updates at a constant stride, whole 256-column tiles and whole
    64-wide K blocks) or one GEMM per update (blocks split at half, rounded up
    to 64)."""
    levels = {}

    def walk(off, s, depth):
        if s <= leaf:
            return
        s1 = ((s // 2 + 63) // 64) * 64
        levels.setdefault(depth, []).append((off, s1, s - s1))
        walk(off, s1, depth + 1)
        walk(off + s1, s - s1, depth + 1)

    walk(0, n, 0)
    count = 1
    for lv in levels.values():
        # with the tensor-core leaves (n a multiple of 64), the leaves carry
        # the updates of at most 2^33 multiply-adds
        if n % 64 == 0:
            lv = [u for u in lv if m * u[1] * u[2] > 2 ** 33]
        if not lv:
            continue
        off0, s1, s2 = lv[0]
        shift = lv[1][0] - off0 if len(lv) > 1 else 0
        batched = (len(lv) > 1 and s1 % 256 == 0 and s2 % 64 == 0 and shift > 0 and
                   all(u == (off0 + k * shift, s1, s2) for k, u in enumerate(lv)))
        count += 1 if batched else len(lv)
    return count


def trmm_flops(spec):
    """Multiply-adds of the triangular product, two flops each: n(n+1)/2 per column."""
    return float(spec["n"]) * (spec["n"] + 1) * spec["m"]


def trsm_launches(n, m=None, leaf=256):
    """Kernel launches of one hgemm_trsm (alpha = 1, out of place): the scaled
    copy, one diagonal solve per leaf and one GEMM per split block. With the
    workspace (leaf=512): the same count over blocks of 512, each leaf one
    product by its inverse (the inverses' launch is counted by the caller)."""
    def count(s):
        if s <= leaf:
            return 1
        s1 = ((s // 2 + 63) // 64) * 64
        return 1 + count(s1) + count(s - s1)
    return 1 + count(n)


def trsm_flops(spec):
    """Back substitution per column: n(n-1)/2 multiply-adds and n divisions, n^2 flops."""
    return float(spec["n"]) * spec["n"] * spec["m"]


# The triangular operations: the call, its oracle, its flop count and launches.
TRI_OPS = {
    "trmm": dict(call="hgemm_trmm", oracle="trmm", flops=trmm_flops, launches=trmm_launches,
                 kernel="hgemm_tri_leaves_tc_kernel, or hgemm_tri_leaves_split_kernel (each leaf unit's K split "
                        "over a cluster) when few leaf units run (hgemm_tri_leaves_kernel when n % 64 != 0) "
                        "+ hgemm update kernels"),
    "trsm": dict(call="hgemm_trsm", oracle="trsm", flops=trsm_flops, launches=trsm_launches,
                 kernel="scale_copy_kernel + trsm_inverse_kernel + hgemm_tc2_kernel (diagonal blocks by their "
                        "inverses, updates); without a workspace trsm_leaf_kernel for the diagonal blocks"),
    "trsm_n": dict(call="hgemm_trsm_op", oracle="trsm_n", flops=trsm_flops, launches=trsm_launches,
                   kernel="scale_copy_kernel + trsm_inverse_kernel + hgemm_tc2(w)_kernel (products by the "
                          "inverses' transposes, updates with N-contiguous A21^T); without a workspace "
                          "trsm_leaf_kernel (forward) for the diagonal blocks"),
}


# hgemm_trsm_last_schedule's values, by name (bench.py reports the schedule a
# solve took), and the kernels of the one-launch schedule.
SCHEDULE_NAMES = {1: "substitution", 2: "recursive (products by the inverses and GEMM updates, one launch each)",
                  4: "chain, fused plan (the inverses' launch, then one persistent cooperative launch, "
                     "one phase per diagonal block)",
                  5: "chain, split plan (the inverses' launch, then one persistent cooperative launch, "
                     "a product phase and an update phase per diagonal block)"}
CHAIN_KERNELS = ("trsm_inverse_kernel (the inverses of the diagonal blocks of 512) + trsm_chain_kernel (one "
                 "persistent cooperative launch: X := B, then per block its product by the inverse and the "
                 "update of every block still to be solved, grid barriers between the phases)")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other configurations after the 8192-cube headline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="target wall time of a whole --impl reference run")
    ap.add_argument("--a-layout", choices=["row", "col"], default="row",
                    help="A stored M x K row-major (the default) or K x M (column-major)")
    ap.add_argument("--b-layout", choices=["col", "row"], default="col",
                    help="B stored N x K (column-major, the default) or K x N row-major")
    ap.add_argument("--no-workspace", action="store_true",
                    help="TRSM workloads: hgemm_trsm without a workspace (substitution for every diagonal block)")
    ap.add_argument("--epilogue", choices=sorted(EPILOGUES), default="none",
                    help="fused epilogue through hgemm_ex (default: the plain product)")
    ap.add_argument("--force-path", choices=sorted(FORCED_PATHS), default="auto",
                    help="profiling aid, GEMM workloads: run the product on this kernel (hgemm_force_path) "
                         "instead of the one the library chooses")
    return ap.parse_args()


# hgemm_force_path values by name (the HGEMM_PATH_* constants of hgemm.h)
FORCED_PATHS = {"auto": -1, "tc": 2, "skinny": 3, "generic": 4, "pair": 5, "wide": 6, "narrow": 7}


# Fused epilogues of hgemm_ex: (alpha, beta, with bias, relu). bias_relu is the
# kernel-fusion example of the CUDA chapter (matmul + bias + ReLU);
# accumulate is C += A·B (the update step of a recursive TRMM).
EPILOGUES = {"none": None, "bias_relu": (1.0, 0.0, True, True), "accumulate": (1.0, 1.0, False, False),
             "accumulate_bias_relu": (1.0, 1.0, True, True)}


# ------------------------------------------------------------------- helpers

def flops_of(spec):
    return 2.0 * spec["M"] * spec["N"] * spec["K"]


def bytes_of(spec, epilogue=None):
    """Algorithmic bytes: A and B read once, C written once; plus C read once
    when beta != 0 and the bias read once."""
    M, N, K = spec["M"], spec["N"], spec["K"]
    extra = 0.0
    if epilogue:
        alpha, beta, with_bias, relu = epilogue
        extra = (2.0 * M * N if beta != 0 else 0.0) + (2.0 * N if with_bias else 0.0)
    return 2.0 * (M * K + N * K + M * N) + extra


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The source file of each kernel; with the shared headers and the build
# flags it determines the compiled kernel, so a recorded ncu traffic figure
# stays valid while their hash is unchanged.
KERNEL_SOURCES = {"hgemm_tc_kernel": ("hgemm_tc.cu",), "hgemm_tc2_kernel": ("hgemm_tc2.cu",),
                  "hgemm_tc2w_kernel": ("hgemm_tc2w.cu",), "hgemm_skinny_kernel": ("hgemm_skinny.cu",),
                  "hgemm_generic_kernel": ("hgemm_generic.cu",),
                  "trsm_chain_kernel": ("hgemm_trsm_chain.cu", "trsm_chain.h"),
                  "hgemm_tri_leaves_tc_kernel": ("hgemm_trileaf.cu",),
                  "hgemm_tri_leaves_split_kernel": ("hgemm_trileaf.cu",)}
SHARED_SOURCES = ["internal.h", "kernel_common.cuh", "ptx.cuh", "debug.cuh"]


def kernel_sources_sha(kernel):
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "tensor_core_dense_fp16_gb300")
    files = [os.path.join(pkg, "csrc", n) for n in SHARED_SOURCES]
    for name in KERNEL_SOURCES.get(kernel, ()):
        files.append(os.path.join(pkg, "csrc", name))
    files.append(os.path.join(pkg, "build.py"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, sha):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (a `traffic_record:` JSON line in profiles/)."""
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path, encoding="utf-8") as f:
            for line in f:
                m = re.match(r"\s*traffic_record:\s*(\{.*\})\s*$", line)
                if not m:
                    continue
                try:
                    rec = json.loads(m.group(1))
                except ValueError:
                    continue
                if (rec.get("kernel") == kernel and rec.get("workload") == workload
                        and rec.get("source_sha") == sha):
                    return float(rec["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t_start = time.time()

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    except ValueError:
                        continue
                    rows.append([ts.timestamp()] + parts[2:])
        os.unlink(self.path)
        # keep the samples taken inside the timed region, widened by one
        # sampling period so that a short region still gets one
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        use = inside or rows[-3:]
        sm = [float(r[1]) for r in use if _num(r[1])]
        smax = [float(r[2]) for r in use if _num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "power_w_max": max((float(r[3]) for r in use if _num(r[3])), default=None)}


def _num(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


class NvmlSampler:
    """In-process, read-only NVML sampling (libnvidia-ml through ctypes) of
    the SM clock, board power and clock-event reasons, about every
    millisecond in a background thread, so that even a region of a few
    milliseconds gets samples while the kernels run. Changes no setting."""

    NVML_CLOCK_SM = 1
    # nvmlClocksEventReason* bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid, period_s=0.001):
        import ctypes
        import threading
        self.ct = ctypes
        self.period = period_s
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.error = None
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            self.handle = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
                raise OSError(f"no NVML device with UUID {uuid}")
            self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = (float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
                self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0 else None)
        except (OSError, AttributeError) as e:
            self.lib = None
            self.error = str(e)

    def _run(self):
        ct = self.ct
        clk, mw, why = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag.is_set():
            t = time.perf_counter()
            ok = self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ct.byref(clk)) == 0
            pw = self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw)) == 0
            rs = self.reason_fn(self.handle, ct.byref(why)) == 0
            if ok:
                self.samples.append((t, float(clk.value), mw.value / 1000.0 if pw else None,
                                     int(why.value) if rs else 0))
            time.sleep(self.period)

    def start(self):
        import threading
        if self.lib is None:
            return
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self, t0, t1):
        """Summary of the samples taken between perf_counter times t0 and t1."""
        if self.lib is None:
            return {"source": "nvml unavailable", "error": self.error, "samples": 0}
        self.stop_flag.set()
        self.thread.join(timeout=2)
        self.lib.nvmlShutdown()
        use = [r for r in self.samples if t0 <= r[0] <= t1]
        sm = [r[1] for r in use]
        power = [r[2] for r in use if r[2] is not None]
        reasons = sorted({name for r in use for bit, name in self.REASONS.items() if r[3] & bit})
        return {"source": f"nvml, every {self.period * 1e3:.0f} ms inside the timed region",
                "sm_mhz": statistics.median(sm) if sm else None,
                "sm_mhz_min": min(sm) if sm else None, "sm_mhz_max": max(sm) if sm else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(use),
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None}


def nvsmi_id(torch, dev, local):
    """An nvidia-smi --id for this process's GPU (nvidia-smi ignores
    CUDA_VISIBLE_DEVICES, so prefer the device UUID)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def reduce_max(value, dist, device):
    """The largest `value` over all ranks (the slowest rank's time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, steps, flops, max_total_ms):
    """Work of all ranks (each ran `steps` products of `flops`) over the
    slowest rank's time for them."""
    return world * steps * flops / (max_total_ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def timed_region(torch, dev, local, stream, step, flush, steps, dist):
    """Times `steps` calls of step(), each after an L2 flush (outside the
    events) and bracketed by CUDA events on `stream`, between barriers, while
    NVML (in-process, ~1 ms) and nvidia-smi (20 ms) sample the clocks.
    Returns (per-call times in ms, clock summary)."""
    gpu_id = nvsmi_id(torch, dev, local)
    smi = ClockSampler(gpu_id)
    nv = NvmlSampler(gpu_id)
    smi.start()
    nv.start()
    time.sleep(0.15)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    switch = sys.getswitchinterval()
    sys.setswitchinterval(0.0005)   # let the sampling thread in while the loop launches
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0, p0 = time.time(), time.perf_counter()
    for s_ev, e_ev in evs:
        flush.zero_()
        s_ev.record(stream)
        step()
        e_ev.record(stream)
    torch.cuda.synchronize(dev)
    t1, p1 = time.time(), time.perf_counter()
    sys.setswitchinterval(switch)
    if dist:
        dist.barrier()
    clocks = nv.stop(p0, p1)
    clocks["nvidia_smi"] = smi.stop(t0, t1)
    if not clocks.get("sm_mhz"):
        for key in ("sm_mhz", "sm_max_mhz", "reasons", "power_w_max"):
            clocks[key] = clocks["nvidia_smi"].get(key)
    return [s_ev.elapsed_time(e_ev) for s_ev, e_ev in evs], clocks


# The other configurations of the problem, timed after the headline in the
# default run with the same protocol (L2 flush before each launch, CUDA
# events on the launching stream, median).
CONFIG_WORKLOADS = ["hgemm_256", "hgemm_256_int", "hgemm_2048", "hgemm_1000_ragged",
                    "hgemm_4096x256x4096_skinny"]
KERNEL_OF_PATH = {2: "hgemm_tc_kernel", 7: "hgemm_tc_kernel", 5: "hgemm_tc2_kernel",
                  6: "hgemm_tc2w_kernel", 3: "hgemm_skinny_kernel", 4: "hgemm_generic_kernel"}
TILES_OF_PATH = {2: "128x256", 7: "128x64", 5: "256x256 pairs", 6: "256x512 pairs",
                 3: "split K", 4: "generic"}


def roofline_of(flops, nbytes, ms, peaks):
    """Roofline time = the slower of the flops at the dense FP16 peak and the
    bytes at HBM bandwidth; fraction = roofline time / measured time."""
    peak = peaks["bf16_tflops"] * FP16_PER_BF16
    t_tensor = flops / (peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    return {"bound": bound, "frac": max(t_tensor, t_hbm) / (ms * 1e-3),
            "tflops": flops / (ms * 1e-3) / 1e12, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "roofline_us": 1e6 * max(t_tensor, t_hbm)}


def time_launch_floor(torch, tc, dev, stream, flush, launches=200, warmup=5):
    """The fixed cost of one launch under the same protocol: a kernel that
    does nothing, in the pair kernel's launch configuration, after an L2
    flush, bracketed by CUDA events."""
    for _ in range(warmup):
        flush.zero_()
        tc.hgemm_launch_floor(True, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(launches)]
    torch.cuda.synchronize(dev)
    for s_ev, e_ev in evs:
        flush.zero_()
        s_ev.record(stream)
        tc.hgemm_launch_floor(True, stream)
        e_ev.record(stream)
    torch.cuda.synchronize(dev)
    times = [s_ev.elapsed_time(e_ev) for s_ev, e_ev in evs]
    return {"kernel": "hgemm_launch_floor (empty kernel, the pair kernel's launch configuration)",
            "launches": launches, "ms_median": statistics.median(times),
            "ms_mean": statistics.fmean(times), "ms_min": min(times)}


def time_configs(torch, tc, dev, stream, flush, peaks, launches=50, warmup=5, floor_ms=None):
    """Each configuration: `launches` flushed, event-timed calls of hgemm.
    With the launch floor, also the fraction of (roofline + floor) time."""
    out = {}
    for name in CONFIG_WORKLOADS:
        a, b, spec = synth.workload(name)
        M, N, K = spec["M"], spec["N"], spec["K"]
        da = torch.from_numpy(a).to(dev)
        db = torch.from_numpy(b).to(dev)
        dc = torch.empty((M, N), dtype=torch.float16, device=dev)
        path = tc.hgemm_select_path(da, db, dc, M, N, K)
        for _ in range(warmup):
            flush.zero_()
            tc.hgemm(da, db, dc, M, N, K, stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(launches)]
        torch.cuda.synchronize(dev)
        for s_ev, e_ev in evs:
            flush.zero_()
            s_ev.record(stream)
            tc.hgemm(da, db, dc, M, N, K, stream)
            e_ev.record(stream)
        torch.cuda.synchronize(dev)
        if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
            raise RuntimeError(f"a kernel wait timed out timing {name}")
        times = [s_ev.elapsed_time(e_ev) for s_ev, e_ev in evs]
        med = statistics.median(times)
        rec = {"M": M, "N": N, "K": K, "seed": spec["seed"], "values": spec["kind"],
               "launches": launches, "ms_median": med, "ms_mean": statistics.fmean(times),
               "ms_min": min(times), "path": KERNEL_OF_PATH.get(path, f"path {path}"),
               "tiles": TILES_OF_PATH.get(path, "?")}
        rec.update(roofline_of(flops_of(spec), bytes_of(spec), med, peaks))
        if floor_ms is not None:
            rec["frac_with_floor"] = (rec["roofline_us"] * 1e-3 + floor_ms) / med
        rec["traffic"] = profiled_traffic(rec["path"], name, kernel_sources_sha(rec["path"]))
        out[name] = rec
    return out


# ------------------------------------------------------------ the oracle leg

def oracle_sample(spec, a, b, target_s, nthreads):
    """Times the oracle on whole rows of C: returns (flops, seconds, rows)."""
    import oracle
    N, K = spec["N"], spec["K"]
    # calibrate on one row per thread, then size the sample to target_s
    rows = min(nthreads, spec["M"])
    t = time.perf_counter()
    oracle.hgemm(a[:rows], b, nthreads=nthreads)
    dt = time.perf_counter() - t
    if dt < target_s:
        scale = max(1, int(target_s / max(dt, 1e-6)))
        rows = min(spec["M"], rows * scale)
        t = time.perf_counter()
        oracle.hgemm(a[:rows], b, nthreads=nthreads)
        dt = time.perf_counter() - t
    return 2.0 * rows * N * K, dt, rows


def run_reference(args, spec, a, b, world, rank):
    if rank != 0:
        return 0
    if spec.get("op") in TRI_OPS:
        return run_tri_reference(args, spec, a, b, world)
    nthreads = os.cpu_count() or 1
    per_step = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    import oracle
    oracle.build()
    N, K = spec["N"], spec["K"]
    rows = min(nthreads, spec["M"])
    t = time.perf_counter()
    oracle.hgemm(a[:rows], b, nthreads=nthreads)
    dt = time.perf_counter() - t
    base = rows
    rows = min(spec["M"], int(rows * per_step / max(dt, 1e-6)))
    rows = max(base, rows - rows % base)  # whole rows, a multiple of the thread count
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        oracle.hgemm(a[:rows], b, nthreads=nthreads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    total = sum(times)
    value = 2.0 * rows * N * K * len(times) / total / 1e12
    sample = (f"{rows} whole rows of C per step ({rows}x{N} outputs, K={K}) of the "
              f"{args.workload} workload; FP64 oracle, {nthreads} threads")
    line = {
        "impl": "reference", "metric": metric_for(args.workload, spec), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}",
                   "M": spec["M"], "N": spec["N"], "K": spec["K"], "seed": spec["seed"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def tri_oracle_columns(op, a_col, b_col, cols, nthreads):
    """The oracle's triangular product or solve on the first `cols` columns of B."""
    import oracle
    return getattr(oracle, TRI_OPS[op]["oracle"])(a_col.T, b_col[:cols].T, nthreads=nthreads)


def run_tri_reference(args, spec, a_col, b_col, world):
    import oracle
    oracle.build()
    op = spec["op"]
    nthreads = os.cpu_count() or 1
    n, m = spec["n"], spec["m"]
    per_step = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    cols = min(m, nthreads)
    t = time.perf_counter()
    tri_oracle_columns(op, a_col, b_col, cols, nthreads)
    dt = time.perf_counter() - t
    cols = max(min(m, nthreads), min(m, int(cols * per_step / max(dt, 1e-6))))
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        tri_oracle_columns(op, a_col, b_col, cols, nthreads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    total = sum(times)
    value = TRI_OPS[op]["flops"](dict(spec, m=cols)) * len(times) / total / 1e12
    sample = (f"the first {cols} columns of B per step (n={n}) of the {args.workload} workload; "
              f"FP64 oracle, {nthreads} threads")
    line = {
        "impl": "reference", "metric": metric_for(args.workload, spec), "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}",
                   "n": n, "m": m, "seed": spec["seed"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_tri_ours(args, spec, a_col, b_col, world, rank, local):
    """The TRMM page's product (hgemm_trmm) or solve (hgemm_trsm): same timing
    protocol as the GEMM workloads (L2 flushed before every timed call)."""
    import torch
    import tensor_core_dense_fp16_gb300 as tc

    tc.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    n, m = spec["n"], spec["m"]
    op = spec["op"]
    ops = TRI_OPS[op]
    flops = ops["flops"](spec)
    call = getattr(tc, ops["call"])
    stream = torch.cuda.current_stream(dev)
    da = torch.from_numpy(a_col).to(dev)
    db = torch.from_numpy(b_col).to(dev)
    dc = torch.empty((m, n), dtype=torch.float16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)

    if op == "trsm" and not args.no_workspace:
        # caller-owned workspace for the diagonal blocks' inverses, allocated once
        work = torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device=dev)

        def step():
            tc.hgemm_trsm_ws(da, n, db, n, dc, n, n, m, 1.0, work, None, stream)
    elif op == "trsm_n":
        work = (None if args.no_workspace else
                torch.empty(tc.hgemm_trsm_workspace_size(n), dtype=torch.uint8, device=dev))

        def step():
            tc.hgemm_trsm_op(tc.HGEMM_OP_N, da, n, db, n, dc, n, n, m, 1.0, work, None, stream)
    else:
        def step():
            call(da, n, db, n, dc, n, n, m, 1.0, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
        raise RuntimeError("a kernel wait timed out during warm-up")
    # the solve's schedule (hgemm_trsm_ws picks it from the shape)
    schedule = tc.hgemm_trsm_last_schedule() if op in ("trsm", "trsm_n") else None
    chain = schedule in (tc.HGEMM_TRSM_CHAIN_FUSED, tc.HGEMM_TRSM_CHAIN_SPLIT)
    times_ms, clocks = timed_region(torch, dev, local, stream, step, flush, args.steps, dist)
    if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
        raise RuntimeError("a kernel wait timed out in the timed region")
    # value and roofline from the median call (the slowest rank's median)
    median_ms = reduce_max(statistics.median(times_ms), dist, dev)
    mean_ms = reduce_max(statistics.fmean(times_ms), dist, dev)
    value = whole_job_tflops(world, 1, flops, median_ms)

    e2e = None
    if not args.no_e2e:
        ha = torch.from_numpy(a_col).pin_memory()
        hb = torch.from_numpy(b_col).pin_memory()
        hc = torch.empty((m, n), dtype=torch.float16).pin_memory()
        e_steps = max(3, min(args.steps, 10))

        def e2e_step():
            da.copy_(ha, non_blocking=True)
            db.copy_(hb, non_blocking=True)
            step()
            hc.copy_(dc, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e_ev.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = reduce_max(s_ev.elapsed_time(e_ev), dist, dev)
        e2e = {"value": whole_job_tflops(world, e_steps, flops, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": 2 * (n * n + n * m), "d2h_bytes_per_step": 2 * n * m,
               "ms_per_step": e_ms / e_steps}

    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"] * FP16_PER_BF16
    achieved = flops / (median_ms * 1e-3) / 1e12
    # DRAM traffic of the solve's dominant launch (the chain kernel), or of a
    # TRMM that is one launch of the leaves, from a committed ncu record of the
    # current sources, per launch
    traffic, traffic_kernel = None, None
    if chain:
        traffic_kernel = "trsm_chain_kernel"
    elif op == "trmm" and n % 64 == 0 and trmm_launches(n, m) == 1:
        for k in ("hgemm_tri_leaves_split_kernel", "hgemm_tri_leaves_tc_kernel"):
            if profiled_traffic(k, args.workload, kernel_sources_sha(k)) is not None:
                traffic_kernel = k
                break
    if traffic_kernel:
        traffic = profiled_traffic(traffic_kernel, args.workload, kernel_sources_sha(traffic_kernel))
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "traffic_kernel": traffic_kernel,
            "peak_source": f"{peak_src}: bf16_tflops (burst) x {FP16_PER_BF16} fp16/bf16",
            "timing": "median call", "kernel": CHAIN_KERNELS if chain else ops["kernel"],
            "algorithmic_flops": flops, "algorithmic_bytes": 2.0 * (n * (n + 1) / 2 + 2 * n * m)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        cols = min(m, nthreads)
        t = time.perf_counter()
        tri_oracle_columns(op, a_col, b_col, cols, nthreads)
        dt = time.perf_counter() - t
        if dt < args.cpu_seconds:
            cols = min(m, max(cols, int(cols * args.cpu_seconds / max(dt, 1e-6))))
            t = time.perf_counter()
            tri_oracle_columns(op, a_col, b_col, cols, nthreads)
            dt = time.perf_counter() - t
        cpu = {"value": ops["flops"](dict(spec, m=cols)) / dt / 1e12, "unit": UNIT, "cores": nthreads,
               "kind": "oracle",
               "sample": f"the first {cols} columns of B (n={n}) of the {args.workload} workload "
                         f"in {dt:.1f} s; FP64 oracle, {nthreads} threads"}
    if rank == 0:
        line = {
            "metric": metric_for(args.workload, spec), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": median_ms,
            "ms_per_step_mean": mean_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}",
                       "n": n, "m": m, "seed": spec["seed"],
                       "l2": "flushed before every timed call (write of 2x L2 size, outside the events)",
                       "inputs": "resident in HBM",
                       "path": ("hgemm_trsm_ws" if op == "trsm" and not args.no_workspace else
                                "hgemm_trsm_op(N, workspace)" if op == "trsm_n" and not args.no_workspace else
                                ops["call"]),
                       "schedule": SCHEDULE_NAMES.get(schedule),
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * (2 if chain else
                                          (ops["launches"](n, m, 512) + 1)
                                          if op in ("trsm", "trsm_n") and not args.no_workspace
                                          else ops["launches"](n, m)),
            "clocks": dict(clocks, kcycles_per_step=(median_ms * clocks["sm_mhz"]
                                                     if clocks.get("sm_mhz") else None)),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------- our leg

def run_ours(args, spec, a, b, world, rank, local):
    import torch
    import tensor_core_dense_fp16_gb300 as tc

    tc.load()  # fails loudly if the extension is missing
    tc.hgemm_force_path(FORCED_PATHS[args.force_path])
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    M, N, K = spec["M"], spec["N"], spec["K"]
    flops = flops_of(spec)
    stream = torch.cuda.current_stream(dev)

    a_col, b_row = args.a_layout == "col", args.b_layout == "row"
    layouts = a_col or b_row
    # the same values stored in the requested order (A K x M, B K x N)
    da = torch.from_numpy(np.ascontiguousarray(a.T) if a_col else a).to(dev)
    db = torch.from_numpy(np.ascontiguousarray(b.T) if b_row else b).to(dev)
    lda, ldb = (M if a_col else K), (N if b_row else K)
    dc = torch.empty((M, N), dtype=torch.float16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)
    epi = EPILOGUES[args.epilogue]
    if layouts:
        # M- or N-contiguous operands take the path of the same shape in the
        # default layout, except that the single-CTA kernel reads K-major
        # operands only (the pair kernel stands in for it)
        tma = lda % 8 == 0 and ldb % 8 == 0 and N % 8 == 0
        path = tc.hgemm_select_path(da, db, dc, M, N, K) if tma else tc.HGEMM_PATH_GENERIC
        if path in (tc.HGEMM_PATH_TC, tc.HGEMM_PATH_TC_NARROW):
            path = tc.HGEMM_PATH_TC_PAIR
    else:
        path = tc.hgemm_select_path(da, db, dc, M, N, K)
    if epi is not None and path == tc.HGEMM_PATH_TC_WIDE:
        path = tc.HGEMM_PATH_TC_PAIR   # a fused epilogue takes 256x256 tiles there (hgemm.h)
    alpha, beta, with_bias, relu = epi if epi is not None else (1.0, 0.0, False, False)
    dbias = None
    if epi is not None:
        gen = torch.Generator(device="cpu").manual_seed(spec["seed"] + 7)
        dbias = (torch.rand(N, generator=gen) - 0.5).half().to(dev) if with_bias else None
        dc.copy_((torch.rand((M, N), generator=gen) - 0.5).half())
    if layouts:
        a_l = tc.HGEMM_A_COL_MAJOR if a_col else tc.HGEMM_A_ROW_MAJOR
        b_l = tc.HGEMM_B_ROW_MAJOR if b_row else tc.HGEMM_B_COL_MAJOR

        def step():
            tc.hgemm_layout(a_l, b_l, da, lda, db, ldb, dc, N, M, N, K, alpha, beta, dbias, relu,
                            stream)
    elif epi is None:
        def step():
            tc.hgemm(da, db, dc, M, N, K, stream)
    else:
        def step():
            tc.hgemm_ex(da, db, dc, M, N, K, alpha, beta, dbias, relu, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
        raise RuntimeError("a kernel wait timed out during warm-up")

    times_ms, clocks = timed_region(torch, dev, local, stream, step, flush, args.steps, dist)
    if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
        raise RuntimeError("a kernel wait timed out in the timed region")
    # value and roofline from the median launch (the slowest rank's median)
    median_ms = reduce_max(statistics.median(times_ms), dist, dev)
    mean_ms = reduce_max(statistics.fmean(times_ms), dist, dev)
    value = whole_job_tflops(world, 1, flops, median_ms)

    # ---- end to end through the host-buffer entry point (the plain product)
    e2e = None
    if not args.no_e2e and epi is None and not layouts:
        ha = torch.from_numpy(a).pin_memory()
        hb = torch.from_numpy(b).pin_memory()
        hc = torch.empty((M, N), dtype=torch.float16).pin_memory()
        e_steps = max(3, min(args.steps, 20))
        for _ in range(2):
            tc.hgemm_host(ha, hb, hc, M, N, K, da, db, dc, stream)
        torch.cuda.synchronize(dev)
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        s_ev.record(stream)
        for _ in range(e_steps):
            tc.hgemm_host(ha, hb, hc, M, N, K, da, db, dc, stream)
        e_ev.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = reduce_max(s_ev.elapsed_time(e_ev), dist, dev)
        if tc.hgemm_device_status(stream) != tc.HGEMM_OK:
            raise RuntimeError("a kernel wait timed out in the end-to-end run")
        e2e = {"value": whole_job_tflops(world, e_steps, flops, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": 2 * (M * K + N * K), "d2h_bytes_per_step": 2 * M * N,
               "ms_per_step": e_ms / e_steps}

    # ---- roofline of the dominant (only) kernel
    peaks, peak_src = load_peaks()
    kernel = {tc.HGEMM_PATH_TC: "hgemm_tc_kernel", tc.HGEMM_PATH_TC_NARROW: "hgemm_tc_kernel",
              tc.HGEMM_PATH_TC_PAIR: "hgemm_tc2_kernel",
              tc.HGEMM_PATH_TC_WIDE: "hgemm_tc2w_kernel",
              tc.HGEMM_PATH_SKINNY: "hgemm_skinny_kernel",
              tc.HGEMM_PATH_GENERIC: "hgemm_generic_kernel"}.get(path, f"path {path}")
    nbytes = bytes_of(spec, epi)
    ai = flops / nbytes
    ridge = peaks["bf16_tflops"] * FP16_PER_BF16 * 1e12 / (peaks["hbm_gbs"] * 1e9)
    sha = kernel_sources_sha(kernel)
    traffic = profiled_traffic(kernel, args.workload if not layouts else
                               f"{args.workload}+a_{args.a_layout}/b_{args.b_layout}", sha)
    if ai >= ridge:
        peak = peaks["bf16_tflops"] * FP16_PER_BF16
        achieved = flops / (median_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src}: bf16_tflops (burst) x {FP16_PER_BF16} fp16/bf16"}
    else:
        peak = peaks["hbm_gbs"]
        achieved = nbytes / (median_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src}: hbm_gbs"}
    roof.update({"timing": "median launch", "kernel": kernel, "algorithmic_flops": flops,
                 "algorithmic_bytes": nbytes, "source_sha": sha})

    # ---- the other configurations (default run, rank 0)
    configs = None
    if (rank == 0 and args.workload == DEFAULT_WORKLOAD and not args.no_configs and epi is None
            and not layouts):
        floor = time_launch_floor(torch, tc, dev, stream, flush)
        configs = {args.workload: dict({"M": M, "N": N, "K": K, "seed": spec["seed"],
                                        "values": spec["kind"], "launches": args.steps,
                                        "ms_median": median_ms, "ms_mean": mean_ms,
                                        "ms_min": min(times_ms), "path": kernel, "traffic": traffic},
                                       **roofline_of(flops, nbytes, median_ms, peaks))}
        configs[args.workload]["frac_with_floor"] = (
            (configs[args.workload]["roofline_us"] * 1e-3 + floor["ms_median"]) / median_ms)
        configs.update(time_configs(torch, tc, dev, stream, flush, peaks, floor_ms=floor["ms_median"]))
        configs["launch_floor"] = floor

    # ---- the oracle on this host's cores (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        nthreads = os.cpu_count() or 1
        fl, dt, rows = oracle_sample(spec, a, b, args.cpu_seconds, nthreads)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": nthreads, "kind": "oracle",
               "sample": f"{rows} whole rows of C ({rows}x{N} outputs, K={K}) of the "
                         f"{args.workload} workload in {dt:.1f} s; FP64 oracle, "
                         f"{nthreads} threads"}

    if rank == 0:
        line = {
            "metric": metric_for(args.workload, spec), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": median_ms,
            "ms_per_step_mean": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}",
                       "M": M, "N": N, "K": K, "seed": spec["seed"],
                       "l2": "flushed before every timed launch (write of 2x L2 size, "
                             "outside the events)",
                       "inputs": "resident in HBM", "path": kernel,
                       "forced_path": args.force_path,
                       "epilogue": args.epilogue, "a_layout": args.a_layout,
                       "b_layout": args.b_layout,
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": dict(clocks, kcycles_per_step=(median_ms * clocks["sm_mhz"]
                                                     if clocks.get("sm_mhz") else None)),
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference" and rank != 0:
        return 0
    a, b, spec = synth.workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, spec, a, b, world, rank)
    if spec.get("op") in TRI_OPS:
        return run_tri_ours(args, spec, a, b, world, rank, local)
    return run_ours(args, spec, a, b, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
