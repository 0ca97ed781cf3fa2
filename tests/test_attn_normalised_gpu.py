"""The normalised form of the attention forward (o = O~ / l kept after every key
tile: "Online softmax", zerotofrontier.app, "From weights to outputs", the
second way to write it) on the GPU against the float64 oracle.

Bars as for the forward (``bars.py``): the plain 1e-2 on every element of the
full-size workload, 1e-2 + 2^-8 |O_ref| elsewhere; LSE within 1e-3.  The
single-query case is also held against the oracle's own normalised stream.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import check_attention, record

pytestmark = pytest.mark.gpu


def run(case):
    kl = case.key_len.cuda() if case.key_len is not None else None
    o, lse = osm.attn_fwd(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, case.causal,
                          kl, normalised=True)
    assert osm.device_status() == 0
    return o, lse


def ref(case, bh=None):
    kl = case.key_len.numpy() if case.key_len is not None else None
    if bh is None:
        return oracle.attention_ref(W.as_f64(case.q), W.as_f64(case.k), W.as_f64(case.v),
                                    case.scale, case.causal, kl)
    b, h = bh
    return oracle.attention_ref(W.as_f64(case.q[b:b + 1, h:h + 1]),
                                W.as_f64(case.k[b:b + 1, h:h + 1]),
                                W.as_f64(case.v[b:b + 1, h:h + 1]), case.scale, case.causal,
                                None if kl is None else kl[b:b + 1])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 1, 127, 129), (1, 2, 300, 300),
                                   (1, 1, 257, 1000), (2, 2, 1000, 1000)])
def test_shapes(cuda_ok, shape, d, causal):
    B, H, Nq, Nk = shape
    case = W.attention(sum(shape) + d + 5 * causal, B, H, Nq, Nk, d, causal,
                       (max(1, Nk // 3), Nk))
    o, lse = run(case)
    check_attention(W.as_f64(o), W.as_f64(lse), *ref(case))


def test_key_len_edges_and_growing_scores(cuda_ok):
    N = 700
    case = W.attention(61, 4, 2, N, N, 128, True, None)
    case.key_len = torch.tensor([0, 1, N - 1, N], dtype=torch.int32)
    k = case.k.float() * torch.linspace(1.0, 8.0, N).view(1, 1, N, 1)   # maxima keep growing
    case.k = k.to(torch.bfloat16)
    o, lse = run(case)
    check_attention(W.as_f64(o), W.as_f64(lse), *ref(case))
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_single_query_against_the_normalised_stream(cuda_ok):
    """One query row against 4096 keys (bf16 inputs): the GPU's normalised form,
    the oracle's normalised block stream (block 64) and the definition agree."""
    q, k, v, _ = W.single_query(1)
    d = q.shape[0]
    qb, kb, vb = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / d ** 0.5
    o, lse = osm.attn_fwd(qb.view(1, 1, 1, d).cuda(), kb.view(1, 1, -1, d).cuda(),
                          vb.view(1, 1, -1, d).cuda(), scale, False, None, normalised=True)
    assert osm.device_status() == 0
    on, ln = oracle.online_attention_single_normalised(W.as_f64(qb), W.as_f64(kb), W.as_f64(vb),
                                                       scale, 64)
    check_attention(W.as_f64(o).reshape(1, d), W.as_f64(lse).reshape(1), on[None], np.array([ln]))


def test_full_size_noncausal(cuda_ok):
    """B4 H16 N4096 d128: every row of 8 whole heads, plain bar; and against the
    single-division kernel on the whole output."""
    case = W.attn()
    o, lse = run(case)
    eo = el = 0.0
    for b, h in [(b, h) for b in range(4) for h in (0, 15)]:
        ro, rl = ref(case, (b, h))
        e = check_attention(W.as_f64(o[b:b + 1, h:h + 1]), W.as_f64(lse[b:b + 1, h:h + 1]), ro,
                            rl, plain=True)
        eo, el = max(eo, e[0]), max(el, e[1])
    record("normalised form, attn B4 H16 N4096 d128 (8 whole heads)", o_err=eo, lse_err=el)
    o1, l1 = osm.attn_fwd(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, False, None)
    assert float((o.float() - o1.float()).abs().max()) <= 2e-2
    assert float((lse - l1).abs().max()) <= 1e-4
