import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (seconds to minutes)")


def read_fixture(name):
    """Parse a golden fixture: 'key v1 v2 ...' lines, '#' comments."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _device_bounds_checks():
    """Under the bounds-checked library (LCSW_EXPECT_CHECKS=1, set by
    test_gpu_checks.py for its child run) every test must leave the device
    check words clean."""
    yield
    if os.environ.get("LCSW_EXPECT_CHECKS") == "1":
        import long_context_sparse_weighted_b300 as lcsw
        L = lcsw.lib()
        assert L.lcsw_checks_enabled() == 1, "the bounds-checked library is not the one loaded"
        code = L.lcsw_check_status()
        assert code == 0, f"a device-side bounds check failed (code {code})"
