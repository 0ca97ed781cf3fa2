import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes on the CPU oracle)")


def read_golden(name):
    """Parse a golden fixture: 'key: v1 v2 ...' lines; '#' lines are comments.

    Repeated keys collect into a list of rows.
    """
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            vals = [float(t) for t in rest.replace("|", " ").split()]
            out.setdefault(key.strip(), []).append(vals)
    return {k: (v[0] if len(v) == 1 else v) for k, v in out.items()}


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
