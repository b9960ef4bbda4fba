"""The GPU parity tests again, against the bounds-checked build.

liblcsw_checks.so is the same source compiled with -DLCSW_CHECKS=1: the
kernels check their data-dependent indices (candidate positions, selection
lists, histogram bins, output positions) and record a failure in a device
check word instead of trapping.  A child pytest run loads that library
(LCSW_LIBRARY) and, after every test, requires lcsw_check_status() == 0
(tests/conftest.py), besides each test's own comparison with the oracle.
"""
import os
import subprocess
import sys

import pytest

from long_context_sparse_weighted_b300 import _build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_kernels.py", "tests/test_gpu_decode.py", "tests/test_gpu_reuse.py",
          "tests/test_gpu_kda.py", "tests/test_gpu_mla.py", "tests/test_gpu_fp8.py",
          "tests/test_gpu_kv8.py", "tests/test_gpu_kvi8.py"]


def test_parity_suites_pass_under_device_bounds_checks():
    lib = _build.build(checks=True)
    env = dict(os.environ, LCSW_LIBRARY=lib, LCSW_EXPECT_CHECKS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu and not slow",
                        "-p", "no:cacheprovider", *SUITES], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
