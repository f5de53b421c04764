"""Builds libhgemm.so, the C-ABI library, in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``tensor_core_dense_fp16_gb300/_build/libhgemm.so`` with the CUDA runtime
linked statically (the library then loads on hosts without a GPU driver,
and finds the driver lazily when first used).

``build(debug=True)`` (``python -m tensor_core_dense_fp16_gb300.build --debug``)
makes the checking variant ``_build/debug/libhgemm.so`` with -DHGEMM_DEBUG
(device-side range and alignment checks, see csrc/debug.cuh); the binding
loads it when HGEMM_LIBRARY_VARIANT=debug.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libhgemm.so")
DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libhgemm.so")
SOURCES = ["hgemm_api.cu", "hgemm_tc.cu", "hgemm_tc2.cu", "hgemm_tc2w.cu", "hgemm_skinny.cu", "hgemm_generic.cu", "hgemm_trsm.cu",
           "hgemm_trileaf.cu", "hgemm_trsm_chain.cu"]
HEADERS = ["ptx.cuh", "internal.h", "kernel_common.cuh", "debug.cuh", "trsm_chain.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhgemm.so")


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "hgemm.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compiles and links libhgemm.so (debug: the checking variant) if it is
    missing or out of date."""
    lib, out_dir = (DEBUG_LIB, DEBUG_DIR) if debug else (LIB, OUT_DIR)
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []
    if debug:
        extra = extra + ["-DHGEMM_DEBUG"]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
