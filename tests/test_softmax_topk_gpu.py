"""Fused softmax + top-k on the GPU against the float64 oracle.

Indices are compared exactly (the order -- value descending, then column
ascending -- is total, so the answer is unique); probabilities within 1e-5
relative (the softmax bar), plus 1e-37 absolute for terms below the fp32
normal range, which the kernel flushes to 0.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def check(x_cpu, k, idx, prob, rows=None):
    x64 = W.as_f64(x_cpu)
    if rows is not None:
        x64 = x64[rows]
        idx, prob = idx[rows], prob[rows]
    ri, rp = oracle.softmax_topk_ref(x64, k)
    gi = idx.cpu().numpy().astype(np.int64)
    gp = W.as_f64(prob)
    assert np.array_equal(gi, ri)
    assert np.all(np.abs(gp - rp) <= 1e-5 * rp + 1e-37)


SHAPES = [(1, 1), (3, 5), (7, 31), (4, 1000), (2, 4097), (5, 32768), (2, 100003), (3, 262144)]


@pytest.mark.parametrize("k", [1, 2, 3, 8, 16, 32])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(cuda_ok, shape, k):
    rows, cols = shape
    if k > cols:
        pytest.skip("k > cols")
    x = W.softmax_logits(seed=70 + cols % 97, rows=rows, cols=cols)  # 1% of entries tie at 40.0
    idx, prob = osm.softmax_topk(x.cuda(), k)
    check(x, k, idx, prob)


def test_ties_masked_entries_and_empty_rows(cuda_ok):
    rng = np.random.default_rng(71)
    x = rng.integers(-4, 5, size=(6, 3000)).astype(np.float32)   # heavy ties
    x[1, ::2] = -np.inf
    x[2, :] = -np.inf                                             # an all -inf row
    x[3, :] = 1.5                                                 # all equal
    x[4, :2990] = -np.inf                                         # only 10 finite entries
    xt = torch.from_numpy(x)
    for k in (1, 7, 16, 32):
        idx, prob = osm.softmax_topk(xt.cuda(), k)
        check(xt, k, idx, prob)
        assert torch.equal(idx[2].cpu(), torch.arange(k, dtype=torch.int32))
        assert torch.all(prob[2] == 0)


def test_monotone_rows(cuda_ok):
    """Rows sorted ascending (every later entry beats the list so far) and
    descending (the first entries are the answer), on the vector path and
    split over a cluster."""
    for cols in (4096, 1 << 19):
        up = torch.arange(cols, dtype=torch.float32) / cols
        x = torch.stack([up, up.flip(0), up * 0 + 0.25, up.roll(cols // 3)])
        for k in (2, 16, 32):
            idx, prob = osm.softmax_topk(x.cuda(), k)
            check(x, k, idx, prob)
            assert torch.equal(idx[0].cpu(), torch.arange(cols - 1, cols - 1 - k, -1, dtype=torch.int32))
            assert torch.equal(idx[1].cpu(), torch.arange(k, dtype=torch.int32))


def test_unaligned_and_odd_widths(cuda_ok):
    """The scalar path: a row length that is not a multiple of 4 and a view that
    starts one element into its buffer."""
    x = W.softmax_logits(seed=72, rows=9, cols=1001)
    idx, prob = osm.softmax_topk(x.cuda(), 8)
    check(x, 8, idx, prob)
    buf = torch.zeros(4 * 2048 + 1)
    buf[1:] = W.softmax_logits(seed=73, rows=4, cols=2048).reshape(-1)
    xv = buf.cuda()[1:].view(4, 2048)
    idx, prob = osm.softmax_topk(xv, 5)
    check(buf[1:].view(4, 2048), 5, idx, prob)


def test_cluster_split_rows(cuda_ok):
    """Few long rows: each row is split over a cluster of CTAs."""
    x = W.softmax_logits(seed=74, rows=2, cols=1 << 20)
    x[1, (1 << 20) - 1] = 100.0          # the best entry in the last CTA's slice
    idx, prob = osm.softmax_topk(x.cuda(), 32)
    check(x, 32, idx, prob)
    assert int(idx[1, 0]) == (1 << 20) - 1


def test_group_filter_edge_rows(cuda_ok):
    """The second pass reads again only the groups of 16 entries whose maximum
    reaches the warp's threshold.  Rows where most groups do (heavy ties, all
    equal), where a thread's groups share a slot (slices longer than 16 steps
    of the first pass), where the few finite entries are spread over those
    shared slots, and where the best entries sit in the ragged last group of
    the last slice."""
    cols = (1 << 20) + 12
    rng = np.random.default_rng(76)
    x = rng.integers(-4, 5, size=(4, cols)).astype(np.float32)   # ties: most groups hold a 4
    x[1, :] = -np.inf
    x[1, rng.choice(cols, 40, replace=False)] = rng.normal(size=40).astype(np.float32)
    x[2, :] = 0.5                                                 # all equal
    x[3] = rng.normal(size=cols).astype(np.float32)
    x[3, cols - 3:] = [50.0, 60.0, 70.0]
    xt = torch.from_numpy(x)
    for k in (2, 8, 32):
        idx, prob = osm.softmax_topk(xt.cuda(), k)
        check(xt, k, idx, prob)
        assert torch.equal(idx[2].cpu(), torch.arange(k, dtype=torch.int32))
        assert idx[3, 0] == cols - 1 and idx[3, 1] == cols - 2


@pytest.mark.parametrize("k", [2, 8, 16, 32])
def test_rows_without_ties(cuda_ok, k):
    """2 N(0,1) entries with no repeated spike value: the group filter and the
    candidate rounds on continuous data, rows of one CTA and of a cluster."""
    for rows, cols in ((64, 32768), (3, 1 << 19)):
        x = W.softmax_logits(seed=77 + k, rows=rows, cols=cols, spike_frac=0.0)
        idx, prob = osm.softmax_topk(x.cuda(), k)
        check(x, k, idx, prob)


def test_full_size_rows(cuda_ok):
    """4096 x 32768 softmax workload (2 N(0,1), 1% of entries = 40.0), k = 8:
    every row's indices exactly, probabilities within the bar."""
    x = W.softmax_logits(2)
    idx, prob = osm.softmax_topk(x.cuda(), 8)
    assert osm.device_status() == 0
    check(x, 8, idx, prob)


def test_deterministic(cuda_ok):
    x = W.softmax_logits(seed=75, rows=64, cols=50000).cuda()
    a = osm.softmax_topk(x, 16)
    b = osm.softmax_topk(x, 16)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
