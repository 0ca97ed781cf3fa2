"""The library compiled with OSM_CHECKED: its kernels check the global indices
they compute (an index out of range is recorded as OSM_ERR_INDEX and the
access skipped).  Every operation on small and edge shapes must run without a
single report and still match the oracle.  The checked library is built here
and exercised in a process of its own (tests/checked_cases.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_no_index_fault(cuda_ok):
    from exact_tiled_attention_osm_gb300 import build
    lib = build.build(checked=True)
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py"), lib],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    assert "checked build clean" in r.stdout
