"""Host-side logic of the benchmark (CPU only): the roofline arithmetic of
each configuration and the clock sampler's behaviour without a GPU."""

import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PEAKS = {"hbm_gbs": 6789.0, "bf16_tflops": 1874.3}


def test_roofline_tensor_bound_8192_cube():
    spec = dict(M=8192, N=8192, K=8192)
    flops, nbytes = bench.flops_of(spec), bench.bytes_of(spec)
    assert flops == 2.0 * 8192 ** 3
    assert nbytes == 2.0 * 3 * 8192 ** 2
    r = bench.roofline_of(flops, nbytes, 0.6, PEAKS)
    assert r["bound"] == "tensor"
    # 1.0995e12 flop at 1874.3 TFLOP/s = 586.6 us; measured 600 us
    assert r["roofline_us"] == pytest.approx(flops / 1874.3e12 * 1e6)
    assert r["frac"] == pytest.approx(flops / 1874.3e12 / 0.6e-3)
    assert r["tflops"] == pytest.approx(flops / 0.6e-3 / 1e12)


def test_roofline_hbm_bound_skinny():
    spec = dict(M=4096, N=256, K=4096)
    flops, nbytes = bench.flops_of(spec), bench.bytes_of(spec)
    assert nbytes == 37748736.0
    r = bench.roofline_of(flops, nbytes, 0.0209, PEAKS)
    assert r["bound"] == "hbm"
    assert r["roofline_us"] == pytest.approx(nbytes / 6789e9 * 1e6)   # 5.56 us
    assert r["frac"] == pytest.approx(nbytes / 6789e9 / 20.9e-6)      # 0.266
    assert r["gbs"] == pytest.approx(nbytes / 20.9e-6 / 1e9)


def test_fused_epilogue_bytes():
    spec = dict(M=64, N=32, K=16)
    plain = bench.bytes_of(spec)
    assert bench.bytes_of(spec, (1.0, 1.0, True, False)) == plain + 2 * 64 * 32 + 2 * 32
    assert bench.bytes_of(spec, (2.0, 0.0, False, True)) == plain


def test_config_list_covers_the_other_workloads():
    import synth
    assert set(bench.CONFIG_WORKLOADS) <= set(synth.WORKLOADS)
    assert bench.DEFAULT_WORKLOAD not in bench.CONFIG_WORKLOADS
    names = {"hgemm_256", "hgemm_256_int", "hgemm_2048", "hgemm_1000_ragged",
             "hgemm_4096x256x4096_skinny"}
    assert set(bench.CONFIG_WORKLOADS) == names


def test_nvml_sampler_without_a_device_reports_itself_unavailable():
    s = bench.NvmlSampler("GPU-00000000-0000-0000-0000-000000000000")
    s.start()
    rec = s.stop(0.0, 1.0)
    if s.lib is None:
        assert rec["samples"] == 0 and "unavailable" in rec["source"]
    else:   # a host with a GPU: whatever it sampled is summarised
        assert rec["samples"] >= 0


def test_path_tables_match_the_header():
    """The benchmark's names for the kernel paths agree with hgemm.h."""
    import tensor_core_dense_fp16_gb300 as tc
    paths = {"tc": tc.HGEMM_PATH_TC, "skinny": tc.HGEMM_PATH_SKINNY, "generic": tc.HGEMM_PATH_GENERIC,
             "pair": tc.HGEMM_PATH_TC_PAIR, "wide": tc.HGEMM_PATH_TC_WIDE, "narrow": tc.HGEMM_PATH_TC_NARROW}
    assert bench.FORCED_PATHS == dict(paths, auto=-1)
    assert set(bench.KERNEL_OF_PATH) == set(paths.values()) == set(bench.TILES_OF_PATH)
    # each kernel a path names has its sources listed for the traffic records
    assert set(bench.KERNEL_OF_PATH.values()) <= set(bench.KERNEL_SOURCES)


def test_traffic_records_are_well_formed():
    """Every traffic_record line of profiles/ parses, names a kernel whose
    sources the benchmark hashes and a known workload, and carries a 16-digit
    hash and a positive byte count."""
    import glob
    import json
    import os
    import re
    import synth
    found = 0
    for path in sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md"))):
        with open(path, encoding="utf-8") as f:
            for line in f:
                m = re.match(r"\s*traffic_record:\s*(\{.*\})\s*$", line)
                if not m:
                    continue
                rec = json.loads(m.group(1))
                found += 1
                assert rec["kernel"] in bench.KERNEL_SOURCES, (path, rec)
                assert rec["workload"].split("+")[0] in synth.WORKLOADS, (path, rec)
                assert re.fullmatch(r"[0-9a-f]{16}", rec["source_sha"]), (path, rec)
                assert rec["bytes_per_launch"] > 0, (path, rec)
    assert found >= 8


@pytest.mark.parametrize("workload", ["hgemm_256", "trsm_n_4096x256"])
def test_reference_arm_line(workload):
    """`bench.py --impl reference` (the oracle on this host's cores) prints one
    JSON line with the GPU arm's metric, unit and direction, a bounded sample
    described in cpu_baseline, and an e2e of its own value with no copies."""
    import json
    import subprocess
    import sys

    import synth
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "2", "--warmup", "1"],
                         check=True, capture_output=True, text=True, timeout=600, cwd=ROOT).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    spec = synth.WORKLOADS[workload]
    assert d["impl"] == "reference"
    assert d["metric"] == bench.metric_for(workload, spec)
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith(workload)
