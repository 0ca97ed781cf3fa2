"""Attention forward on the GPU against the float64 oracle.

Bars (``bars.py``; BF16 inputs, float64 oracle on the same bf16-rounded inputs):
  O:   |O_gpu - O_ref| <= 1e-2 on every element of the full-size workloads;
       elsewhere <= 1e-2 + 2^-8 |O_ref| (1e-2 on the value before the output's
       own bf16 storage rounding, which alone can reach 2^-8 |O|);
  LSE: |lse_gpu - lse_ref| <= 1e-3, and -inf exactly where the oracle has -inf;
  masked keys contribute exactly zero (bitwise test across two paddings).
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import check_attention, record

pytestmark = pytest.mark.gpu


def check(o, lse, ro, rl, plain=False):
    return check_attention(W.as_f64(o), W.as_f64(lse), ro, rl, plain)


def run(case, dev="cuda"):
    kl = case.key_len.to(dev) if case.key_len is not None else None
    o, lse = osm.attn_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.scale, case.causal,
                          kl)
    assert osm.device_status() == 0
    return o, lse


def oracle_of(case, rows=None, bh=None):
    q, k, v = case.q, case.k, case.v
    kl = case.key_len.numpy() if case.key_len is not None else None
    if bh is not None:  # restrict to a list of (b, h)
        outs = [oracle.attention_ref(W.as_f64(q[b:b + 1, h:h + 1]), W.as_f64(k[b:b + 1, h:h + 1]),
                                     W.as_f64(v[b:b + 1, h:h + 1]), case.scale, case.causal,
                                     None if kl is None else kl[b:b + 1], rows=rows)
                for b, h in bh]
        return outs
    return oracle.attention_ref(W.as_f64(q), W.as_f64(k), W.as_f64(v), case.scale, case.causal,
                                kl, rows=rows)


SHAPES = [(1, 1, 1, 1), (1, 1, 63, 63), (1, 2, 64, 64), (1, 1, 65, 65), (2, 1, 127, 129),
          (1, 1, 129, 127), (1, 2, 300, 300), (1, 1, 256, 256), (1, 1, 257, 1000),
          (1, 1, 1000, 257), (2, 2, 513, 513), (1, 1, 1, 4097), (1, 1, 4097, 4097)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(cuda_ok, shape, causal):
    B, H, Nq, Nk = shape
    case = W.attention(sum(shape) + 100 * causal, B, H, Nq, Nk, 128, causal, (max(1, Nk // 3), Nk))
    o, lse = run(case)
    check(o, lse, *oracle_of(case))


@pytest.mark.parametrize("causal", [False, True])
def test_key_len_edges(cuda_ok, causal):
    N = 300
    case = W.attention(21, 4, 2, N, N, 128, causal, None)
    case.key_len = torch.tensor([0, 1, N - 1, N], dtype=torch.int32)
    o, lse = run(case)
    ro, rl = oracle_of(case)
    check(o, lse, ro, rl)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    # one visible key: O = v_0 exactly (weight 1, bf16 value reproduced exactly)
    v0 = case.v[1, :, 0:1, :].to(o.device).expand(-1, N, -1)
    assert torch.equal(o[1], v0)


def test_no_keys_and_more_queries_than_keys(cuda_ok):
    case = W.attention(22, 1, 2, 100, 0, 128, False, None)
    o, lse = run(case)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    case = W.attention(23, 2, 1, 400, 150, 128, True, None)   # causal, Nq > Nk
    o, lse = run(case)
    check(o, lse, *oracle_of(case))
    assert torch.all(torch.isneginf(lse[:, :, :250]))


def test_masked_keys_contribute_exactly_zero(cuda_ok):
    """Keys past key_len hold two different finite garbage patterns; O and LSE
    must be bitwise identical (and the causal future likewise)."""
    B, H, N = 2, 2, 700
    case = W.attention(24, B, H, N, N, 128, True, (200, 650))
    outs = []
    for pattern in range(2):
        k, v = case.k.clone(), case.v.clone()
        for b in range(B):
            L = int(case.key_len[b])
            if pattern == 0:
                k[b, :, L:] = 1e30
                v[b, :, L:] = -1e30
            else:
                g = torch.Generator().manual_seed(b)
                k[b, :, L:] = (torch.randn(k[b, :, L:].shape, generator=g) * 100).to(torch.bfloat16)
                v[b, :, L:] = (torch.randn(v[b, :, L:].shape, generator=g) * 100).to(torch.bfloat16)
        c2 = W.AttnCase(case.q, k, v, case.scale, True, case.key_len)
        outs.append(run(c2))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    check(*outs[0], *oracle_of(case))


@pytest.mark.parametrize("causal", [False, True])
def test_growing_scores(cuda_ok, causal):
    """Scores whose row maximum keeps growing from tile to tile: moderate growth
    (the reference is raised by a few binades, already-formed terms rescaled),
    and jumps so large that everything before them underflows to zero."""
    B, H, N = 2, 2, 1000
    case = W.attention(23, B, H, N, N, 128, causal, (700, N))
    k = case.k.float()
    grow = torch.linspace(1.0, 12.0, N).view(1, 1, N, 1)      # steady growth
    k = k * grow
    k[0, :, 600] *= 40.0     # one huge key in a late tile (batch 0)
    k[1, 1, 300:310] *= 25.0  # a block of large keys mid-row
    case.k = k.to(torch.bfloat16)
    o, lse = run(case)
    eo, el = check(o, lse, *oracle_of(case))
    record(f"growing scores causal={causal}", o_err=eo, lse_err=el)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_sharp_rows(cuda_ok, causal, d):
    """Queries scaled by 10: nearly one-hot rows whose dominant weight is not
    a power of two against the lazy reference.  O is normalised by the sum of
    the bf16 weights the P V product used, so the dominant weight's own
    rounding cancels: the storage bar holds with no allowance for the weights'
    rounding."""
    case = W.attention(78 + d, 3, 4, 1024, 1024, d, causal, None)
    case.q = (case.q.float() * 10.0).to(torch.bfloat16)
    o, lse = run(case)
    eo, el = check(o, lse, *oracle_of(case))
    record(f"sharp rows q*10 d{d} causal={causal}", o_err=eo, lse_err=el)


@pytest.mark.parametrize("bounded", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_dominant_key_in_a_late_tile(cuda_ok, d, causal, bounded):
    """Every query is beta times one key of a late key tile (beta in [1, 4]),
    values of magnitude 4 to 6: rows are one-hot to within e^-8 .. e^-30, the
    dominant weight is 2^k f against the reference the row's first tile set
    (raised by whole binades when it would pass 2^16).  Plain bar everywhere;
    and where the oracle's output equals the dominant key's value to 1e-4,
    the GPU's output is that bf16 value exactly."""
    B, H, N = 2, 3, 1024
    case = W.attention_dominant_keys(300 + d + 2 * causal, B, H, N, d, causal)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    bound = None
    if bounded:
        bound = case.scale * float(case.q.float().norm(dim=-1).max()) * float(
            case.k.float().norm(dim=-1).max())
    o, lse = osm.attn_fwd(q, k, v, case.scale, causal, None, score_bound=bound)
    assert osm.device_status() == 0
    ro, rl = oracle_of(case)
    eo, el = check(o, lse, ro, rl)
    record(f"dominant key d{d} causal={causal} bounded={bounded}", o_err=eo, lse_err=el)
    vt = W.as_f64(case.v)[:, :, case.meta["target"], :]
    onehot = np.all(np.abs(ro - vt) <= 1e-4, axis=-1)
    assert onehot.mean() > 0.25
    og = W.as_f64(o)
    assert np.array_equal(og[onehot], vt[onehot])


@pytest.mark.parametrize("causal", [False, True])
def test_scores_far_below_zero(cuda_ok, causal):
    """Every score near -200: against the starting reference 0 all terms would
    underflow, so the first chunk of each row lowers the reference."""
    B, H, N = 1, 2, 700
    case = W.attention(24, B, H, N, N, 128, causal, (400, N))
    q = 4.0 + 0.05 * case.q.float()
    k = -4.5 + 0.05 * case.k.float()
    case.q, case.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    o, lse = run(case)
    ro, rl = oracle_of(case)
    assert float(np.max(rl[np.isfinite(rl)])) < -150
    check(o, lse, ro, rl)


def qk_normed(seed, causal):
    """QK-norm inputs: q and k rows scaled to norm sqrt(d), so |s| <= scale * d."""
    B, H, N = 2, 2, 1000
    case = W.attention(seed, B, H, N, N, 128, causal, (500, N))
    for name in ("q", "k"):
        t = getattr(case, name).float()
        t = t / t.norm(dim=-1, keepdim=True) * 128 ** 0.5
        setattr(case, name, t.to(torch.bfloat16))
    nq = float(case.q.float().norm(dim=-1).max())
    nk = float(case.k.float().norm(dim=-1).max())
    return case, case.scale * nq * nk   # an upper bound of every score


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("which", ["valid", "too_low", "far_too_high"])
def test_known_bound(cuda_ok, causal, which):
    """Scores with a known bound (QK-norm): exact whatever the bound -- a valid
    one, one far below the scores (the reference is raised) and one so far
    above them that every term would underflow (the reference is lowered)."""
    case, bound = qk_normed(25 + causal, causal)
    bound = {"valid": bound, "too_low": -60.0, "far_too_high": bound + 400.0}[which]
    kl = case.key_len.cuda()
    o, lse = osm.attn_fwd(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, causal, kl,
                          score_bound=bound)
    assert osm.device_status() == 0
    check(o, lse, *oracle_of(case))


def test_deterministic(cuda_ok):
    case = W.attention(25, 2, 4, 1000, 1000, 128, True, (500, 1000))
    a, b = run(case), run(case)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_full_size_noncausal(cuda_ok):
    """B4 H16 N4096 d128, non-causal: every row of 16 whole heads (four per
    batch entry) against the oracle; the whole output finite."""
    case = W.attn()
    o, lse = run(case)
    eo = el = 0.0
    for b in range(4):
        for h in (0, 5, 10, 15):
            (ro, rl), = oracle_of(case, bh=[(b, h)])
            e = check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ro, rl, plain=True)
            eo, el = max(eo, e[0]), max(el, e[1])
    record("attn B4 H16 N4096 d128 (16 whole heads)", o_err=eo, lse_err=el)
    assert torch.all(torch.isfinite(o)) and torch.all(torch.isfinite(lse))


def test_full_size_causal_padded(cuda_ok):
    """B8 H32 N8192 d128, causal, key_len ~ U[4096, 8192]: every row of 8 heads
    -- the shortest and the longest batch entries and two more, heads 0 and
    31 -- against the oracle; the whole output finite."""
    case = W.attn_causal()
    o, lse = run(case)
    kl = case.key_len.numpy()
    bs = [int(np.argmin(kl)), int(np.argmax(kl))]
    bs += [b for b in (0, 7, 1, 6) if b not in bs][:2]
    eo = el = 0.0
    for b in bs:
        for h in (0, 31):
            (ro, rl), = oracle_of(case, bh=[(b, h)])
            e = check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ro, rl, plain=True)
            eo, el = max(eo, e[0]), max(el, e[1])
    record("attn causal+padding B8 H32 N8192 d128 (8 whole heads)", o_err=eo, lse_err=el)
    assert torch.all(torch.isfinite(o)) and torch.all(torch.isfinite(lse))


def test_long_sequence_causal_padded(cuda_ok):
    """One head pair with 32768 keys (256 key tiles per work item), causal,
    key_len 20000 and 32768: sampled rows, including the diagonal tiles' edges
    and rows past key_len."""
    B, H, N = 2, 2, 32768
    case = W.attention(91, B, H, N, N, 128, True, None)
    case.key_len = torch.tensor([20000, 32768], dtype=torch.int32)
    o, lse = run(case)
    rows = np.array([0, 1, 127, 128, 4095, 19999, 20000, 20001, 32767])
    ro, rl = oracle_of(case, rows=rows)
    check(o[:, :, rows], lse[:, :, rows], ro, rl)


def test_very_long_sequence(cuda_ok):
    """131072 queries and keys in one head (1024 key tiles per row at the end),
    causal, and the same head against 131072 keys without a mask for 256
    queries: sampled rows at the start, at tile edges and at the end."""
    N = 131072
    case = W.attention(92, 1, 1, N, N, 128, True, None)
    o, lse = run(case)
    rows = np.array([0, 1, 255, 256, 65535, 65536, N - 129, N - 128, N - 1])
    ro, rl = oracle_of(case, rows=rows)
    check(o[:, :, rows], lse[:, :, rows], ro, rl)
    cross = W.attention(93, 1, 1, 256, N, 128, False, None)
    o, lse = run(cross)
    ro, rl = oracle_of(cross)
    check(o, lse, ro, rl)


def test_many_small_heads(cuda_ok):
    """B·H = 16384 heads of 100 queries and keys (one ragged 128-wide tile
    each): 16384 work items over the persistent grid, causal, d = 64."""
    B, H, N, d = 4096, 4, 100, 64
    g = torch.Generator().manual_seed(94)  # one draw for all heads (fast at this count)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16) for _ in range(3))
    case = W.AttnCase(q, k, v, 1.0 / math.sqrt(d), True, None)
    o, lse = run(case)
    check(o, lse, *oracle_of(case))


def test_cross_attention_shapes(cuda_ok):
    """Nq != Nk without a causal mask (cross-attention): 512 queries against
    16384 keys, and 3000 queries against 200 keys."""
    for seed, (Nq, Nk) in ((92, (512, 16384)), (93, (3000, 200))):
        case = W.attention(seed, 1, 2, Nq, Nk, 128, False, (Nk // 2, Nk))
        o, lse = run(case)
        check(o, lse, *oracle_of(case))


D64_SHAPES = [(1, 1, 1, 1), (1, 2, 65, 65), (2, 1, 127, 129), (1, 2, 300, 300), (1, 1, 257, 1000),
              (2, 2, 1000, 1000)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", D64_SHAPES)
def test_head_dim_64(cuda_ok, shape, causal):
    """d = 64: one 64-column TMA box per tile, N = 64 P.V products."""
    B, H, Nq, Nk = shape
    case = W.attention(sum(shape) + 300 + 7 * causal, B, H, Nq, Nk, 64, causal,
                       (max(1, Nk // 3), Nk))
    o, lse = run(case)
    check(o, lse, *oracle_of(case))


def test_head_dim_64_edges_and_bound(cuda_ok):
    N = 300
    case = W.attention(95, 4, 2, N, N, 64, True, None)
    case.key_len = torch.tensor([0, 1, N - 1, N], dtype=torch.int32)
    o, lse = run(case)
    check(o, lse, *oracle_of(case))
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ob, lb = osm.attn_fwd(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, True,
                          case.key_len.cuda(), score_bound=3.0)
    assert osm.device_status() == 0
    check(ob, lb, *oracle_of(case))


def test_cross_check_torch_sdpa(cuda_ok):
    """Secondary cross-check (not the oracle): torch's scaled_dot_product_attention
    on the same bf16 tensors, causal and with a padding mask; both sides round
    to bf16, so they agree to a few bf16 ulps of O."""
    import torch.nn.functional as F
    for causal in (False, True):
        case = W.attention(96 + causal, 2, 4, 1024, 1024, 128, causal, (600, 1024))
        q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
        kl = case.key_len.cuda()
        o, _ = osm.attn_fwd(q, k, v, case.scale, causal, kl)
        assert osm.device_status() == 0
        j = torch.arange(1024, device="cuda")
        mask = (j[None, :] < kl[:, None])[:, None, None, :]
        if causal:
            mask = mask & (j[None, :] <= j[:, None])[None, None]
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=case.scale)
        err = (o.float() - ref.float()).abs()
        assert float(err.max()) <= 2e-2
        assert float(err.mean()) <= 2e-3
