"""The -DHGEMM_DEBUG build (CPU only): the predicates its device-side checks
use decide values inside and just outside their ranges correctly, and the
checking variant compiles, loads and exports the whole C ABI."""

import ctypes
import re

import pytest

import tensor_core_dense_fp16_gb300 as tc
from tensor_core_dense_fp16_gb300 import build


def test_check_predicates_on_planted_values():
    tc.load()
    assert tc.hgemm_debug_selftest() == 0
    assert tc.hgemm_debug_build() == 0   # the release library carries no checks


def test_debug_variant_builds_and_exports_the_abi():
    lib_path = build.build(debug=True)
    lib = ctypes.CDLL(lib_path)
    lib.hgemm_debug_build.restype = ctypes.c_int
    lib.hgemm_debug_selftest.restype = ctypes.c_int
    assert lib.hgemm_debug_build() == 1
    assert lib.hgemm_debug_selftest() == 0
    with open(build.os.path.join(build.INCLUDE, "hgemm.h"), encoding="utf-8") as f:
        names = re.findall(r"HGEMM_API\s+[\w\s\*]+?\b(hgemm\w*)\s*\(", f.read())
    assert len(names) > 20
    for name in names:
        assert hasattr(lib, name), name
