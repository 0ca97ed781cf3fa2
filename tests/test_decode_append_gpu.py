"""Incremental decode (running summaries extended by appended keys) on the GPU
against the float64 oracle.

Appending keys is one more merge into the stored summary, so after any
sequence of appends the state must be the summary of all keys seen and the
output must equal attention over them.  Bars as for split decode: FP32 O and
LSE within 1e-5; BF16 the storage bar of ``bars.py`` (O within
1e-2 + 2^-8 |O_ref|; LSE within 1e-3).
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import o_bar

pytestmark = pytest.mark.gpu


def oracle_prefix(case, ends):
    """(o, lse) of attention over keys [0, ends[b]) and the float64 summaries."""
    q64, k64, v64 = W.as_f64(case.q), W.as_f64(case.k), W.as_f64(case.v)
    ro, rl = oracle.attention_ref(q64, k64, v64, case.scale, False, np.asarray(ends))
    B, H = q64.shape[:2]
    summ = {}
    for b in range(B):
        for h in range(H):
            n = int(ends[b])
            sc = case.scale * (k64[b, h, :n] @ q64[b, h, 0])
            summ[b, h] = oracle.summary_of(sc, v64[b, h, :n])
    return ro[:, :, 0], rl[:, :, 0], summ


def check_out(o, lse, ro, rl, fp32):
    o, lse = W.as_f64(o)[:, :, 0], W.as_f64(lse)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(lse), ~fin)
    if fp32:
        assert float(np.max(np.abs(o - ro))) <= 1e-5
        tol_l = 1e-5
    else:
        assert np.all(np.abs(o - ro) <= o_bar(ro))
        tol_l = 1e-3
    if fin.any():
        assert float(np.max(np.abs(lse[fin] - rl[fin]))) <= tol_l


def check_state(state, summ, fp32):
    m, l, ot = (W.as_f64(t) for t in state)
    for (b, h), (sm, sl, so) in summ.items():
        if sm == -math.inf:
            assert m[b, h] == -math.inf and l[b, h] == 0 and np.all(ot[b, h] == 0)
            continue
        tol_m = (1e-5 if fp32 else 1e-3) * max(1.0, abs(sm))
        assert abs(m[b, h] - sm) <= tol_m
        # summaries taken at different references differ by a common factor;
        # compare at the oracle's reference
        f = math.exp(m[b, h] - sm)
        assert abs(l[b, h] * f - sl) <= 1e-4 * sl
        assert np.max(np.abs(ot[b, h] * f - so)) <= 1e-3 * sl


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 5, 64])
def test_appends_equal_attention_over_the_prefix(cuda_ok, dtype, d, splits):
    B, H, Nk = 3, 2, 3000
    case = W.decode(seed=50 + d + splits, B=B, H=H, Nk=Nk, d=d, len_range=(Nk, Nk),
                    num_splits=splits)
    q, k, v = (t.to(dtype).cuda() for t in (case.q, case.k, case.v))
    case.q, case.k, case.v = (t.to(dtype) for t in (case.q, case.k, case.v))
    # per-batch boundaries: empty appends, a single key, ragged steps, the whole cache
    bounds = np.array([[0, 0, 0], [1, 0, 7], [1, 129, 7], [17, 130, 1000],
                       [500, 2047, 1001], [2999, 2048, 2600], [3000, 3000, 3000]], np.int32)
    state = osm.decode_state(B, H, d, "cuda")
    ws = torch.empty(osm.decode_append_workspace_bytes(B, H, d, splits), dtype=torch.uint8,
                     device="cuda")
    fp32 = dtype == torch.float32
    for i in range(1, len(bounds)):
        ks = torch.from_numpy(bounds[i - 1]).cuda()
        ke = torch.from_numpy(bounds[i]).cuda()
        o, lse = osm.attn_decode_append(q, k, v, state, ks, ke, case.scale, splits, workspace=ws)
        assert osm.device_status() == 0
        ro, rl, summ = oracle_prefix(case, bounds[i])
        check_out(o, lse, ro, rl, fp32)
        check_state(state, summ, fp32)


def test_empty_append_leaves_state_bitwise(cuda_ok):
    B, H, Nk, d = 2, 3, 600, 128
    case = W.decode(seed=60, B=B, H=H, Nk=Nk, d=d, len_range=(Nk, Nk), num_splits=4)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    state = osm.decode_state(B, H, d, "cuda")
    half = torch.full((B,), 300, dtype=torch.int32, device="cuda")
    o1, l1 = osm.attn_decode_append(q, k, v, state, None, half, case.scale, 4)
    before = [t.clone() for t in state]
    o2, l2 = osm.attn_decode_append(q, k, v, state, half, half, case.scale, 4)
    assert osm.device_status() == 0
    for a, b in zip(before, state):
        assert torch.equal(a, b)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_state_from_the_oracle_is_extended(cuda_ok):
    """A state written from the oracle's own summary of keys [0, a) (fp32), then
    extended on the GPU by [a, L), gives attention over [0, L): the state's
    convention (natural-log max, unnormalised o~) is the pages' summary."""
    B, H, Nk, d = 2, 2, 2000, 128
    case = W.decode(seed=61, B=B, H=H, Nk=Nk, d=d, len_range=(1500, Nk), num_splits=8)
    a = np.array([700, 0], np.int32)
    L = case.key_len.numpy()
    _, _, summ = oracle_prefix(case, a)
    m = torch.tensor([[summ[b, h][0] for h in range(H)] for b in range(B)], dtype=torch.float32)
    l = torch.tensor([[summ[b, h][1] for h in range(H)] for b in range(B)], dtype=torch.float32)
    ot = torch.tensor(np.array([[summ[b, h][2] for h in range(H)] for b in range(B)]),
                      dtype=torch.float32)
    state = (m.cuda(), l.cuda(), ot.cuda())
    o, lse = osm.attn_decode_append(case.q.cuda(), case.k.cuda(), case.v.cuda(), state,
                                    torch.from_numpy(a).cuda(), case.key_len.cuda(), case.scale, 8)
    assert osm.device_status() == 0
    ro, rl, _ = oracle_prefix(case, L)
    check_out(o, lse, ro, rl, False)


def test_matches_split_decode(cuda_ok):
    """One append from the empty state over [0, L) is split decode over L."""
    case = W.decode(seed=62, B=4, H=8, Nk=4096, d=128, len_range=(1, 4096), num_splits=16)
    q, k, v, kl = case.q.cuda(), case.k.cuda(), case.v.cuda(), case.key_len.cuda()
    state = osm.decode_state(4, 8, 128, "cuda")
    o1, l1 = osm.attn_decode_append(q, k, v, state, None, kl, case.scale, 16)
    o2, l2 = osm.attn_decode_splitkv(q, k, v, case.scale, kl, 16)
    assert osm.device_status() == 0
    assert float((o1.float() - o2.float()).abs().max()) <= 2.0 ** -7
    assert float((l1 - l2).abs().max()) <= 1e-5
