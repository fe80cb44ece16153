import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Non-comment lines of a golden fixture, split into tokens."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test: no bounded device-side wait gave up during it.  A
    wait that gives up skips its CTA's stores, so the status word -- not only the
    tolerance check on stale memory -- must show it."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import ternary_weight_linear_02_gb300 as tl
    if tl._lib is None:
        return
    torch.cuda.synchronize()
    code = tl.device_status(clear=True)
    assert code == 0, f"device status {tl.status_string(code)} after {request.node.nodeid}"
