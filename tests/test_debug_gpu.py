"""Small cases on every path under the -DHGEMM_DEBUG build, in a process of
their own (the variant is chosen when the library is loaded): parity with the
oracle and no device-side check or watchdog code (GPU only)."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_path_is_clean_under_the_checks():
    env = dict(os.environ, HGEMM_LIBRARY_VARIANT="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "every path clean" in r.stdout
