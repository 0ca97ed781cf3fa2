"""Pins for the float64 oracle, independent of the oracle itself.

Each test ties an oracle function to something fixed outside it: numbers the
pages print (tests/golden/), closed forms, invariants the pages prove, special
cases with a textbook answer, brute force with exactly rounded sums, and a
library routine (torch softmax / scaled_dot_product_attention in float64).
A deliberately broken merge and deliberately broken attention variants are
planted (in oracle-side code, on the CPU) to show the pins catch such mistakes.
"""
import math
import random

import numpy as np
import pytest
import torch

import oracle as O


# ----------------------------------------------------------------- printed values

def test_p2_tiled_softmax_worked_example(golden):
    g = golden("p2_tiled_softmax.txt")
    row = g["row"]
    tiles = g["tile"]
    want = g["rounded6"]
    naive = O.softmax_rows_ref(np.array(row))
    online = O.tiled_softmax_online(row, tiles)
    assert [round(v, 6) for v in naive] == want
    assert [round(v, 6) for v in online] == want
    # the plain definition with exactly rounded sums agrees too
    assert [round(v, 6) for v in O.softmax_row_fsum(row)] == want


def test_p3_running_max_sum_trace(golden):
    g = golden("p3_running_ml.txt")
    tr = O.online_ml_trace(g["scores"])
    assert tr[0] == (2.0, 1.0)
    assert tr[0] == tuple(g["step1"])
    assert math.exp(tr[0][0] - tr[1][0]) == pytest.approx(g["shrink2"][0], abs=5e-5)
    assert tr[1][0] == g["step2"][0] and tr[1][1] == pytest.approx(g["step2"][1], abs=5e-5)
    assert math.exp(1 - tr[2][0]) == pytest.approx(g["term3"][0], abs=5e-5)
    assert tr[3][0] == g["final"][0] and tr[3][1] == pytest.approx(g["final"][1], abs=5e-5)
    # closed forms of the intermediate sums
    assert tr[1][1] == pytest.approx(math.exp(-3) + 1, rel=1e-15)
    assert tr[2][1] == pytest.approx(math.exp(-3) + 1 + math.exp(-4), rel=1e-15)
    assert tr[3][1] == pytest.approx(math.fsum(math.exp(s - 7) for s in (2, 5, 1, 7)), rel=1e-15)


def test_p3_merge_worked_example(golden):
    g = golden("p3_merge_example.txt")
    va = np.zeros((2, 1))
    vb = np.zeros((2, 1))
    a = O.summary_of(g["half_a_scores"], va)
    b = O.summary_of(g["half_b_scores"], vb)
    assert a[0] == g["half_a"][0] and a[1] == pytest.approx(g["half_a"][1], abs=5e-5)
    assert b[0] == g["half_b"][0] and b[1] == pytest.approx(g["half_b"][1], abs=5e-5)
    assert a[1] * math.exp(a[0] - b[0]) == pytest.approx(g["a_rescaled"][0], abs=5e-5)
    m = O.merge(a, b)
    assert m[1] == pytest.approx(g["merged_l"][0], abs=5e-5)
    # merged == one-score-at-a-time recurrence on the whole row
    full = O.online_ml_trace(g["half_a_scores"] + g["half_b_scores"])[-1]
    assert (m[0], m[1]) == pytest.approx(full, rel=1e-15)


def test_p1_online_equals_naive_single_query(golden):
    g = golden("p1_online_vs_naive.txt")
    d = int(g["shape_q"][0])
    n, _ = (int(x) for x in g["shape_kv"])
    rng = np.random.default_rng(7)
    q, k, v = rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    o_on, lse_on = O.online_attention_single(q, k, v, 1.0, int(g["block"][0]))
    o_def, lse_def = O.attention_ref(q[None, None, None], k[None, None], v[None, None], 1.0)
    # the page prints ~1e-15 for such a draw; we hold both routes to 1e-13
    assert np.max(np.abs(o_on - o_def[0, 0, 0])) < 1e-13
    assert abs(lse_on - lse_def[0, 0, 0]) < 1e-12


# ----------------------------------------------------------------- invariants

@pytest.mark.parametrize("seed", range(5))
def test_running_sum_bounds(seed):
    """1 <= l_j <= j at every step; m_j is the prefix maximum (theorem + bounds)."""
    rng = np.random.default_rng(seed)
    s = rng.standard_normal(300) * rng.uniform(0.5, 30)
    tr = O.online_ml_trace(s)
    for j, (m, l) in enumerate(tr, start=1):
        assert m == np.max(s[:j])
        assert 1.0 - 1e-12 <= l <= j + 1e-9
        assert l == pytest.approx(math.fsum(math.exp(x - m) for x in s[:j]), rel=1e-12)


def test_softmax_against_fsum_and_torch():
    rng = np.random.default_rng(11)
    for n in (1, 2, 3, 7, 64, 1000):
        x = rng.standard_normal(n) * 10
        y = O.softmax_rows_ref(x)
        assert np.allclose(y, O.softmax_row_fsum(list(x)), rtol=1e-14, atol=0)
        assert np.allclose(y, torch.softmax(torch.from_numpy(x), 0).numpy(), rtol=1e-13, atol=0)
        assert math.fsum(y) == pytest.approx(1.0, abs=1e-14)
    # huge logits: the safe form does not overflow (unsafe exp(1000) would)
    y = O.softmax_rows_ref(np.array([1000.0, 999.0, -1000.0]))
    assert np.all(np.isfinite(y)) and y[0] == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    # a fully masked row is defined as zeros
    assert np.all(O.softmax_rows_ref(np.full((2, 5), -np.inf)) == 0)
    # a single finite entry among -inf
    y = O.softmax_rows_ref(np.array([-np.inf, 3.0, -np.inf]))
    assert list(y) == [0.0, 1.0, 0.0]


# ----------------------------------------------------------------- merge algebra

def _rand_summaries(rng, n, dv):
    s = rng.standard_normal(n) * 4
    vals = rng.standard_normal((n, dv))
    return s, vals


def _exact_summary(s, vals, idx):
    """(m, l, o~) of a subset with exactly rounded sums."""
    m = max(s[i] for i in idx)
    w = [math.exp(s[i] - m) for i in idx]
    l = math.fsum(w)
    o = np.array([math.fsum(w[t] * vals[i, c] for t, i in enumerate(idx))
                  for c in range(vals.shape[1])])
    return m, l, o


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_merge_every_order_and_grouping(n):
    """Every ordered set partition, merged left to right, gives the whole set's summary."""
    rng = np.random.default_rng(100 + n)
    s, vals = _rand_summaries(rng, n, 3)
    want = _exact_summary(s, vals, list(range(n)))
    for blocks in O.all_orders_and_groupings(n):
        parts = [O.summary_of(s[b], vals[b]) for b in blocks]
        got = O.merge_all(parts)
        assert got[0] == want[0]
        assert got[1] == pytest.approx(want[1], rel=4 * 2.2e-16 * n)
        assert np.allclose(got[2], want[2], rtol=1e-14, atol=1e-15)


def test_merge_grouping_n7_balanced_vs_left():
    rng = np.random.default_rng(7)
    s, vals = _rand_summaries(rng, 7, 4)
    want = _exact_summary(s, vals, list(range(7)))
    for part in O.set_partitions(range(7)):
        parts = [O.summary_of(s[b], vals[b]) for b in part]
        while len(parts) > 1:  # balanced tree
            parts = [O.merge(parts[i], parts[i + 1]) if i + 1 < len(parts) else parts[i]
                     for i in range(0, len(parts), 2)]
        got = parts[0]
        assert got[0] == want[0]
        assert got[1] == pytest.approx(want[1], rel=1e-14)
        assert np.allclose(got[2], want[2], rtol=1e-13, atol=1e-15)


def test_merge_identity_and_one_step_special_case():
    ident = (O.NEG_INF, 0.0, np.zeros(2))
    a = (1.5, 2.0, np.array([0.3, -1.0]))
    for x in (O.merge(a, ident), O.merge(ident, a)):
        assert x[0] == a[0] and x[1] == a[1] and np.array_equal(x[2], a[2])
    both = O.merge(ident, ident)
    assert both[0] == O.NEG_INF and both[1] == 0 and not np.any(np.isnan(both[2]))
    o, lse = O.finalize(both)
    assert lse == O.NEG_INF and np.all(o == 0)
    # processing one score = merging with (s, 1, v)
    rng = np.random.default_rng(3)
    s, vals = _rand_summaries(rng, 10, 2)
    acc = ident
    for j in range(10):
        acc = O.merge(acc, (s[j], 1.0, vals[j]))
        tr = O.online_ml_trace(s[:j + 1])[-1]
        assert acc[0] == tr[0] and acc[1] == pytest.approx(tr[1], rel=1e-14)


def test_lse_form_merge_is_triple_merge():
    rng = np.random.default_rng(5)
    S, rows, d = 5, 4, 3
    s = rng.standard_normal((S, rows, 6)) * 3
    vals = rng.standard_normal((S, rows, 6, d))
    s[2, 1, :] = -np.inf      # an empty piece for one row
    s[:, 3, :] = -np.inf      # a row that is empty everywhere
    o_parts = np.zeros((S, rows, d))
    lse_parts = np.zeros((S, rows))
    for i in range(S):
        for r in range(rows):
            o_parts[i, r], lse_parts[i, r] = O.finalize(O.summary_of(s[i, r], vals[i, r]))
    o, lse = O.lse_merge_ref(o_parts, lse_parts)
    for r in range(rows):
        # the LSE form equals the triple merge of (lse_s, 1, o_s) with l=0 for empty parts
        trip = O.merge_all([(lse_parts[i, r], 0.0 if np.isneginf(lse_parts[i, r]) else 1.0,
                             o_parts[i, r]) for i in range(S)])
        o2, lse2 = O.finalize(trip)
        assert np.allclose(o[r], o2, rtol=1e-14, atol=1e-15)
        assert (lse[r] == lse2) or lse[r] == pytest.approx(lse2, rel=1e-15)
        # and the whole row's direct summary
        o3, lse3 = O.finalize(O.summary_of(s[:, r].reshape(-1), vals[:, r].reshape(-1, d)))
        assert np.allclose(o[r], o3, rtol=1e-13, atol=1e-14)
        assert (lse[r] == lse3) or lse[r] == pytest.approx(lse3, rel=1e-14)
    assert lse[3] == O.NEG_INF and np.all(o[3] == 0)


def test_planted_merge_bug_is_caught():
    """The merge that adds sums without rescaling fails the order-independence pin."""
    def bad_merge(a, b):
        return max(a[0], b[0]), a[1] + b[1], a[2] + b[2]

    rng = np.random.default_rng(9)
    s, vals = _rand_summaries(rng, 4, 2)
    want = _exact_summary(s, vals, [0, 1, 2, 3])
    parts = [O.summary_of(s[[0, 1]], vals[[0, 1]]), O.summary_of(s[[2, 3]], vals[[2, 3]])]
    good = O.merge(*parts)
    bad = bad_merge(*parts)
    assert good[1] == pytest.approx(want[1], rel=1e-14)
    assert bad[1] != pytest.approx(want[1], rel=1e-3)
    # the page's worked example exposes it too: 1.0498 + 1.0025 != 1.1446
    a = O.summary_of([2.0, 5.0], np.zeros((2, 1)))
    b = O.summary_of([1.0, 7.0], np.zeros((2, 1)))
    assert bad_merge(a, b)[1] != pytest.approx(1.1446, abs=5e-3)


# ----------------------------------------------------------------- attention

def _tiny_case(rng, B, H, Nq, Nk, d):
    return (rng.standard_normal((B, H, Nq, d)), rng.standard_normal((B, H, Nk, d)),
            rng.standard_normal((B, H, Nk, d)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 3, 5, 4), (2, 2, 5, 5, 3), (1, 2, 6, 4, 2), (2, 1, 1, 6, 5)])
def test_attention_vs_bruteforce(shape, causal):
    B, H, Nq, Nk, d = shape
    rng = np.random.default_rng(sum(shape) + causal)
    q, k, v = _tiny_case(rng, B, H, Nq, Nk, d)
    key_len = rng.integers(0, Nk + 1, size=B)
    scale = 0.37
    o1, l1 = O.attention_ref(q, k, v, scale, causal, key_len)
    o2, l2 = O.attention_bruteforce(q, k, v, scale, causal, key_len)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-14)
    fin = np.isfinite(l2)
    assert np.array_equal(np.isneginf(l1), np.isneginf(l2))
    assert np.allclose(l1[fin], l2[fin], rtol=1e-13, atol=1e-14)


def test_attention_special_cases():
    rng = np.random.default_rng(1)
    q, k, v = _tiny_case(rng, 1, 1, 4, 7, 3)
    # one visible key: o = v_0, lse = s_0
    o, lse = O.attention_ref(q, k, v, 0.5, False, [1])
    assert np.allclose(o[0, 0], np.repeat(v[0, 0, :1], 4, axis=0), rtol=0, atol=0)
    assert np.allclose(lse[0, 0], 0.5 * (q[0, 0] @ k[0, 0, 0]), rtol=1e-15)
    # identical keys: uniform weights, lse = s + log n
    k2 = np.repeat(k[:, :, :1], 7, axis=2)
    o, lse = O.attention_ref(q, k2, v, 0.5, False)
    assert np.allclose(o[0, 0], np.repeat(v[0, 0].mean(0, keepdims=True), 4, 0), rtol=1e-14)
    assert np.allclose(lse[0, 0], 0.5 * (q[0, 0] @ k[0, 0, 0]) + math.log(7), rtol=1e-14)
    # no visible key at all: o = 0, lse = -inf
    o, lse = O.attention_ref(q, k, v, 0.5, False, [0])
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    # causal with Nq > Nk: rows with no visible key are -inf
    qa, ka, va = _tiny_case(rng, 1, 1, 6, 3, 2)
    o, lse = O.attention_ref(qa, ka, va, 1.0, True)
    assert np.all(np.isneginf(lse[0, 0, :3])) and np.all(np.isfinite(lse[0, 0, 3:]))


def test_attention_masks_equal_truncation():
    """Causal row i == unmasked attention over keys 0..i+Nk-Nq; padding == truncation."""
    rng = np.random.default_rng(2)
    q, k, v = _tiny_case(rng, 2, 1, 5, 8, 4)
    key_len = [8, 3]
    o, lse = O.attention_ref(q, k, v, 1.0, True, key_len)
    for b in range(2):
        for i in range(5):
            n = min(key_len[b], i + 1 + 3)
            ot, lt = O.attention_ref(q[b:b + 1, :, i:i + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 1.0)
            assert np.allclose(o[b, 0, i], ot[0, 0, 0], rtol=1e-14, atol=1e-15)
            assert lse[b, 0, i] == pytest.approx(lt[0, 0, 0], rel=1e-14)


def test_attention_vs_torch_sdpa_float64():
    rng = np.random.default_rng(4)
    q, k, v = _tiny_case(rng, 2, 3, 33, 47, 8)
    for causal in (False, True):
        o, lse = O.attention_ref(q, k, v, 1 / math.sqrt(8), causal)
        if causal:  # torch's is_causal is top-left aligned; build the bottom-right mask
            mask = torch.ones(33, 47, dtype=torch.bool).tril(47 - 33)
            ot = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask)
        else:
            ot = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v))
        assert np.allclose(o, ot.numpy(), rtol=1e-12, atol=1e-13)
    # lse vs torch.logsumexp of the scaled scores
    s = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) / math.sqrt(8)
    _, lse = O.attention_ref(q, k, v, 1 / math.sqrt(8), False)
    assert np.allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-14)


def test_planted_attention_bugs_are_caught():
    """Plausible slips in an attention oracle (transposed operand, dropped scale,
    off-by-one causal mask) each fail the brute-force pin."""
    rng = np.random.default_rng(8)
    q, k, v = _tiny_case(rng, 1, 1, 4, 4, 3)
    o_ok, _ = O.attention_bruteforce(q, k, v, 0.5, True)

    def variant(qq, kk, vv, scale, causal, shift=0):
        s = scale * (qq[0, 0] @ kk[0, 0].T)
        if causal:
            s = np.where(np.arange(4)[None] <= np.arange(4)[:, None] + shift, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        return (p / p.sum(1, keepdims=True)) @ vv[0, 0]

    assert np.allclose(variant(q, k, v, 0.5, True), o_ok[0, 0], rtol=1e-13)
    assert not np.allclose(variant(q, v, k, 0.5, True), o_ok[0, 0], rtol=1e-3)       # K/V swapped
    assert not np.allclose(variant(q, k, v, 1.0, True), o_ok[0, 0], rtol=1e-3)       # scale dropped
    assert not np.allclose(variant(q, k, v, 0.5, True, 1), o_ok[0, 0], rtol=1e-3)    # mask off by one
    assert not np.allclose(variant(q, k, v, 0.5, False), o_ok[0, 0], rtol=1e-3)      # mask dropped


def test_online_single_query_block_sizes():
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal(16), rng.standard_normal((257, 16)), rng.standard_normal((257, 16))
    o_def, lse_def = O.attention_ref(q[None, None, None], k[None, None], v[None, None], 0.25)
    for block in (1, 7, 64, 256, 1000):
        o, lse = O.online_attention_single(q, k, v, 0.25, block)
        assert np.allclose(o, o_def[0, 0, 0], rtol=1e-13, atol=1e-14)
        assert lse == pytest.approx(lse_def[0, 0, 0], rel=1e-14)


# ---------------------------------------------------------------------------
# Fused softmax + top-k ([P3] the `softmax_topk` exercise after "Precision,
# and what can still go wrong"; Milakov & Gimelshein's fused form).


def _topk_bruteforce(row, k):
    """Sort (-x_i, i) with Python's sort; probabilities with math.exp / fsum."""
    n = len(row)
    order = sorted(range(n), key=lambda i: (-row[i], i))[:k]
    finite = [v for v in row if v != -math.inf]
    if not finite:
        return order, [0.0] * k
    mx = max(finite)
    total = math.fsum(math.exp(v - mx) for v in finite)
    return order, [(math.exp(row[i] - mx) / total if row[i] != -math.inf else 0.0)
                   for i in order]


def test_topk_matches_the_pages_naive_formula():
    """On moderate values with no ties, the page's own (unstable) formula
    idx = argsort(-x)[:k], exp(x[idx]) / sum exp(x) is exact enough to pin."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 300)) * 3
    for k in (1, 4, 17, 300):
        idx, prob = O.softmax_topk_ref(x, k)
        for r in range(5):
            naive_idx = np.argsort(-x[r])[:k]
            naive_p = np.exp(x[r][naive_idx]) / np.exp(x[r]).sum()
            assert np.array_equal(idx[r], naive_idx)
            assert np.allclose(prob[r], naive_p, rtol=1e-13, atol=0)


def test_topk_bruteforce_ties_and_masked_entries():
    rng = np.random.default_rng(32)
    x = rng.integers(-3, 4, size=(6, 40)).astype(np.float64)   # many ties
    x[1, ::3] = -np.inf
    x[2, :] = -np.inf                                           # an all -inf row
    x[3, :] = 2.0                                               # all equal
    for k in (1, 3, 8, 40):
        idx, prob = O.softmax_topk_ref(x, k)
        for r in range(6):
            bi, bp = _topk_bruteforce(list(x[r]), k)
            assert list(idx[r]) == bi
            assert np.allclose(prob[r], bp, rtol=1e-14, atol=0)
    idx, prob = O.softmax_topk_ref(x, 40)
    assert list(idx[3]) == list(range(40))                      # ties: lowest index first
    assert np.all(prob[2] == 0)
    assert math.fsum(prob[0]) == pytest.approx(1.0, abs=1e-14)  # k = n: all the mass
    assert np.all(np.diff(prob[0]) <= 0)                        # probabilities non-increasing


def test_topk_is_stable_where_the_naive_formula_overflows():
    x = np.array([[1000.0, 999.0, 998.0, 0.0]])
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.exp(x[0][:2]) / np.exp(x[0]).sum()
    assert np.all(np.isnan(naive))                              # inf / inf
    idx, prob = O.softmax_topk_ref(x, 2)
    assert list(idx[0]) == [0, 1]
    e = np.exp([0.0, -1.0, -2.0, -1000.0])
    assert np.allclose(prob[0], e[:2] / e.sum(), rtol=1e-15)


def test_planted_topk_bugs_are_caught():
    """Plausible slips (ties broken by the higher index, probabilities
    normalised over the k chosen entries only) fail the brute-force pin."""
    x = np.array([[1.0, 3.0, 3.0, 0.5, 2.0]])
    bi, bp = _topk_bruteforce(list(x[0]), 3)
    idx, prob = O.softmax_topk_ref(x, 3)
    assert list(idx[0]) == bi == [1, 2, 4]
    wrong_ties = list(np.lexsort((-np.arange(5), -x[0]))[:3])
    assert wrong_ties != bi
    wrong_norm = np.exp(x[0][bi]) / np.exp(x[0][bi]).sum()
    assert not np.allclose(wrong_norm, bp, rtol=1e-3)
    assert np.allclose(prob[0], bp, rtol=1e-14)


# ---------------------------------------------------------------------------
# Backward ([P3] "From weights to outputs": lse rebuilds the weights).


def _loss_grads_fd(q, k, v, do, scale, causal, key_len, eps=1e-6):
    """Central differences of sum(dO * O) through the forward definition."""
    def loss(qq, kk, vv):
        o, _ = O.attention_ref(qq, kk, vv, scale, causal, key_len)
        return float(np.sum(do * o))

    grads = []
    for which in range(3):
        base = [q, k, v][which]
        g = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape,key_len", [((1, 1, 5, 5, 4), None), ((2, 1, 4, 6, 3), [6, 2]),
                                           ((1, 2, 6, 3, 4), [3]), ((1, 1, 3, 1, 2), None)])
def test_backward_matches_finite_differences(shape, key_len, causal):
    B, H, Nq, Nk, d = shape
    rng = np.random.default_rng(40 + Nq + 7 * causal)
    q, k, v = (rng.standard_normal(s) for s in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d)))
    do = rng.standard_normal((B, H, Nq, d))
    o, lse = O.attention_ref(q, k, v, 0.7, causal, key_len)
    dq, dk, dv = O.attention_bwd_ref(q, k, v, o, lse, do, 0.7, causal, key_len)
    fq, fk, fv = _loss_grads_fd(q, k, v, do, 0.7, causal, key_len)
    for got, want in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7)


def test_backward_matches_autograd_of_the_definition():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    B, H, N, d = 2, 2, 37, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    kl = [29, 37]
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (q, k, v))
    s = 0.35 * tq @ tk.transpose(-1, -2)
    j = torch.arange(N)
    mask = (j[None, :] <= j[:, None])[None, None] & (j[None, None, None, :] < torch.tensor(kl)[:, None, None, None])
    s = s.masked_fill(~mask, float("-inf"))
    out = torch.softmax(s, dim=-1) @ tv
    out.backward(torch.tensor(do))
    o, lse = O.attention_ref(q, k, v, 0.35, True, kl)
    dq, dk, dv = O.attention_bwd_ref(q, k, v, o, lse, do, 0.35, True, kl)
    assert np.allclose(dq, tq.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_backward_rows_without_keys_and_planted_bugs():
    rng = np.random.default_rng(42)
    q, k, v, do = (rng.standard_normal((1, 1, 4, 3)) for _ in range(4))
    # key_len 0: every weight is 0, so every gradient is 0
    o, lse = O.attention_ref(q, k, v, 0.5, False, [0])
    assert np.all(np.isneginf(lse))
    for g in O.attention_bwd_ref(q, k, v, o, lse, do, 0.5, False, [0]):
        assert np.all(g == 0)
    # plausible slips fail the finite-difference pin
    o, lse = O.attention_ref(q, k, v, 0.5, True)
    fq, fk, fv = _loss_grads_fd(q, k, v, do, 0.5, True, None)
    s = 0.5 * q[0, 0] @ k[0, 0].T
    s = np.where(np.arange(4)[None] <= np.arange(4)[:, None], s, -np.inf)
    p = np.exp(s - lse[0, 0][:, None])
    dp = do[0, 0] @ v[0, 0].T
    D = np.sum(do[0, 0] * o[0, 0], axis=1)
    right = 0.5 * (p * (dp - D[:, None])) @ k[0, 0]
    assert np.allclose(right, fq[0, 0], rtol=1e-6, atol=1e-7)
    assert not np.allclose(0.5 * (p * dp) @ k[0, 0], fq[0, 0], rtol=1e-3)        # D dropped
    assert not np.allclose((p * (dp - D[:, None])) @ k[0, 0], fq[0, 0], rtol=1e-3)  # scale dropped
    assert not np.allclose(0.5 * (p * (dp - D[:, None])).T @ k[0, 0], fq[0, 0], rtol=1e-3)  # dS^T
    assert not np.allclose(p @ do[0, 0], fv[0, 0], rtol=1e-3)                       # P not P^T


def test_normalised_form_equals_the_unnormalised_one():
    """[P3] "From weights to outputs": keeping o = O~ / l after every block (the
    original FlashAttention form) is exact too -- against the definition and
    the unnormalised stream, for several block sizes, and a planted slip
    (the old output not weighted by its share l e^{m - m_new} / l_new)."""
    rng = np.random.default_rng(43)
    q, k, v = rng.standard_normal(16), rng.standard_normal((300, 16)), rng.standard_normal((300, 16))
    k[170] *= 6.0                                    # the max jumps mid-stream
    o_def, lse_def = O.attention_ref(q[None, None, None], k[None, None], v[None, None], 0.4)
    for block in (1, 7, 64, 300):
        o_n, lse_n = O.online_attention_single_normalised(q, k, v, 0.4, block)
        o_u, lse_u = O.online_attention_single(q, k, v, 0.4, block)
        assert np.allclose(o_n, o_def[0, 0, 0], rtol=1e-13, atol=1e-14)
        assert np.allclose(o_n, o_u, rtol=1e-13, atol=1e-14)
        assert lse_n == pytest.approx(lse_def[0, 0, 0], rel=1e-14)
    m, l, o = NEG_INF_, 0.0, np.zeros(16)
    for start in range(0, 300, 64):                  # the slip: o_new = o + w V / l_new
        s = 0.4 * (k[start:start + 64] @ q)
        m_new = max(m, s.max())
        shrink = 0.0 if m == NEG_INF_ else np.exp(m - m_new)
        w = np.exp(s - m_new)
        l_new = shrink * l + w.sum()
        o = o + (w @ v[start:start + 64]) / l_new
        m, l = m_new, l_new
    assert not np.allclose(o, o_def[0, 0, 0], rtol=1e-3)


NEG_INF_ = float("-inf")
