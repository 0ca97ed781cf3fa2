"""Row softmax on the GPU against the float64 oracle (bar: max relative error <= 1e-5)."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import record

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5
# fp32 outputs below the normal range are flushed; relative error is measured
# against max(|ref|, FLOOR)
FLOOR = 1e-30


def rel_err(y, ref):
    return float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), FLOOR)))


def run(x):
    y = osm.softmax_rows(x.cuda())
    assert osm.device_status() == 0
    return W.as_f64(y)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 4), (5, 7), (2, 1000), (7, 4096), (3, 4100),
                                       (4, 8192), (3, 8196), (2, 16388), (3, 32768), (2, 65536),
                                       (2, 65540), (2, 131072), (2, 131076),
                                       (1, 200003), (300, 96), (1, 1 << 22), (70000, 64)])
def test_shapes(cuda_ok, rows, cols):
    x = W.softmax_logits(seed=rows * 7 + cols, rows=rows, cols=cols)
    y = run(x)
    ref = oracle.softmax_rows_ref(W.as_f64(x))
    assert rel_err(y, ref) <= REL_TOL


def test_edge_rows(cuda_ok):
    x = torch.randn(6, 4096) * 3
    x[0] = float("-inf")                       # fully masked row -> zeros
    x[1] = float("-inf")
    x[1, 17] = 2.5                             # one finite entry -> one-hot
    x[2] = 7.0                                 # constant row -> uniform
    x[3, ::2] = float("-inf")                  # half masked
    x[4] = torch.linspace(-80, 80, 4096)       # wide range
    x[5, :] = -1e30                            # huge negative but finite
    y = run(x)
    ref = oracle.softmax_rows_ref(W.as_f64(x))
    assert np.all(y[0] == 0)
    assert y[1, 17] == 1.0 and np.count_nonzero(y[1]) == 1
    assert rel_err(y, ref) <= REL_TOL


def test_in_place_and_unaligned(cuda_ok):
    x = W.softmax_logits(seed=5, rows=9, cols=3000).cuda()
    ref = oracle.softmax_rows_ref(W.as_f64(x))
    y = osm.softmax_rows(x, out=x)             # in place
    assert y.data_ptr() == x.data_ptr()
    assert rel_err(W.as_f64(x), ref) <= REL_TOL
    buf = torch.empty(9 * 3000 + 1, device="cuda")
    xu = buf[1:].view(9, 3000)                 # 4-byte aligned only -> generic kernel
    xu.copy_(W.softmax_logits(seed=5, rows=9, cols=3000).cuda())
    yu = osm.softmax_rows(xu)
    assert rel_err(W.as_f64(yu), ref) <= REL_TOL


def test_deterministic(cuda_ok):
    x = W.softmax_logits(seed=8, rows=64, cols=32768).cuda()
    assert torch.equal(osm.softmax_rows(x), osm.softmax_rows(x))


def test_full_size_workload(cuda_ok):
    """4096 x 32768, 2*N(0,1) with 1% of entries at +40: every row against the
    oracle (in blocks of 256 rows), plus sums and signs on every row."""
    x = W.softmax_logits(seed=2)
    xd = x.cuda()
    y = osm.softmax_rows(xd)
    assert osm.device_status() == 0
    worst = 0.0
    for r0 in range(0, 4096, 256):
        ref = oracle.softmax_rows_ref(W.as_f64(x[r0:r0 + 256]))
        worst = max(worst, rel_err(W.as_f64(y[r0:r0 + 256]), ref))
    record("softmax 4096 x 32768 (every row)", rel_err=worst)
    assert worst <= REL_TOL
    s = y.double().sum(1)
    assert torch.all(torch.isfinite(y)) and torch.all(y >= 0)
    assert float((s - 1).abs().max()) <= 1e-4
