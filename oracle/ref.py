"""Float64 CPU oracle for exact softmax attention and the online-softmax merge.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py`` use it.  It shares no code, constants or helpers with the
CUDA library; it takes plain NumPy arrays (the exact values handed to the GPU,
upcast to float64) and returns NumPy arrays.

Sources (three web pages on one subject):
  [P1] "Online Softmax: How FlashAttention Skips the N×N Matrix" (dev.to)
  [P2] "Online softmax" (guide.dupenodi.dev)
  [P3] "Online softmax" (zerotofrontier.app, textbook chapter 12.2)

Where the method reaches a result with a plain definition (softmax of a row,
softmax attention, log-sum-exp) the oracle is that definition written out:
``softmax_rows_ref`` and ``attention_ref``.  The method's own steps (the scalar
running (m, l) recurrence, the blockwise single-query loop, the summary merge)
are written out separately so the pin tests can check them against the
definitions and against the numbers the pages print.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".

Readings of points the pages leave open (the CUDA library takes the same ones):
  * A row whose every score is -inf (a fully masked row) has l = 0; its output
    row is 0 and its log-sum-exp is -inf.  [P3] "Precision" says such a row
    "must be handled explicitly"; this is the finalize of the merge identity
    (-inf, 0, 0) from [P3] "Merging partial results", property 2.
  * Causal masking with Nq != Nk is bottom-right aligned: query i sees key j
    iff j <= i + (Nk - Nq).  Only keys are padded: key j is visible iff
    j < key_len[b].
  * Scores are s = scale * (q . k); the log-sum-exp is of the scaled scores,
    in natural log.
"""
from __future__ import annotations

import itertools
import math
from typing import Iterable, List, Sequence, Tuple

import numpy as np

NEG_INF = float("-inf")

# ---------------------------------------------------------------------------
# Row softmax: the plain three-pass "safe" definition.
# [P3] "Three passes, and why that is a problem"; [P1] "What problem does
# online softmax actually solve?"
# ---------------------------------------------------------------------------


def softmax_rows_ref(x: np.ndarray) -> np.ndarray:
    """Safe softmax of every row of ``x`` in float64, three explicit passes.

    Pass 1: m = max of the row.  Pass 2: e_i = exp(x_i - m), l = sum e_i.
    Pass 3: y_i = e_i / l.  A row that is entirely -inf returns zeros (see the
    module docstring).
    """
    x = np.asarray(x, dtype=np.float64)
    squeeze = x.ndim == 1
    if squeeze:
        x = x[None, :]
    m = np.max(x, axis=1, keepdims=True) if x.shape[1] else np.full((x.shape[0], 1), NEG_INF)
    ref = np.where(np.isneginf(m), 0.0, m)  # an all -inf row: exp(-inf - 0) = 0
    e = np.exp(x - ref)
    l = np.sum(e, axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        y = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    return y[0] if squeeze else y


def softmax_topk_ref(x: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """The k largest entries of every row and their softmax probabilities.

    [P3] "Precision, and what can still go wrong", the `softmax_topk` exercise
    after it (Milakov & Gimelshein's fused softmax plus top-k): the indices of
    the k largest scores, and exp(x_i) / sum_j exp(x_j) at those indices.  The
    page's own version is unstable; here the probabilities are the safe
    softmax of the whole row (``softmax_rows_ref``) read at the chosen indices.
    Order: value descending, equal values by index ascending (one total order,
    so the result is unique).  Returns (idx int64 [R, k], prob float64 [R, k]).
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim == 1:
        x = x[None, :]
    R, n = x.shape
    if not 1 <= k <= n:
        raise ValueError("need 1 <= k <= number of columns")
    y = softmax_rows_ref(x)
    idx = np.empty((R, k), dtype=np.int64)
    prob = np.empty((R, k), dtype=np.float64)
    cols = np.arange(n)
    for r in range(R):
        order = np.lexsort((cols, -x[r]))[:k]   # primary key -x, then the index
        idx[r] = order
        prob[r] = y[r, order]
    return idx, prob


def softmax_row_fsum(xs: Sequence[float]) -> List[float]:
    """Safe softmax of one short row with exactly rounded sums (math.fsum).

    Brute-force counterpart of ``softmax_rows_ref`` for tiny rows.
    """
    m = max(xs)
    e = [math.exp(x - m) for x in xs]
    l = math.fsum(e)
    return [v / l for v in e]


# ---------------------------------------------------------------------------
# The scalar running (m, l) recurrence.
# [P3] "Two numbers that can be updated" and "The recurrence, and a proof that
# it is right"; [P2] "Walking through it".
# ---------------------------------------------------------------------------


def online_ml_trace(scores: Iterable[float]) -> List[Tuple[float, float]]:
    """Run the running-max / running-sum recurrence one score at a time.

    Starts from m_0 = -inf, l_0 = 0.  At step j:
        m_j = max(m_{j-1}, s_j)
        l_j = l_{j-1} * exp(m_{j-1} - m_j) + exp(s_j - m_j)
    The factor exp(m_{j-1} - m_j) is taken as 0 while m_{j-1} = -inf (it
    discards the empty initial sum; [P3] notes e^{-inf} = 0 there).
    Returns [(m_1, l_1), ..., (m_n, l_n)].
    """
    m, l = NEG_INF, 0.0
    out = []
    for s in scores:
        s = float(s)
        m_new = max(m, s)
        if m_new == NEG_INF:  # only -inf seen so far: nothing to sum yet
            out.append((m_new, 0.0))
            continue
        shrink = 0.0 if m == NEG_INF else math.exp(m - m_new)
        l = l * shrink + math.exp(s - m_new)
        m = m_new
        out.append((m, l))
    return out


def tiled_softmax_online(xs: Sequence[float], tiles: Sequence[Sequence[float]]) -> List[float]:
    """Softmax of a row fed tile by tile, keeping rescaled running numerators.

    [P2] "Walking through it": per tile, take the new running max, multiply the
    running sum and every numerator kept so far by exp(m_old - m_new), append
    exp(x - m_new) for the tile's entries, add them to the running sum; divide
    once at the end.  ``xs`` is only used to check that the tiles cover it.
    """
    flat = [float(v) for t in tiles for v in t]
    if flat != [float(v) for v in xs]:
        raise ValueError("tiles must partition the row in order")
    run_m, run_s, numer = NEG_INF, 0.0, []
    for tile in tiles:
        m_new = max([run_m] + [float(v) for v in tile])
        factor = 0.0 if run_m == NEG_INF else math.exp(run_m - m_new)
        numer = [n * factor for n in numer]
        fresh = [math.exp(float(v) - m_new) for v in tile]
        run_s = run_s * factor + sum(fresh)
        numer.extend(fresh)
        run_m = m_new
    return [n / run_s for n in numer]


# ---------------------------------------------------------------------------
# Summaries (m, l, o~) and the merge.
# [P3] "Merging partial results", "The same merge, in log-sum-exp form".
# ---------------------------------------------------------------------------

Summary = Tuple[float, float, np.ndarray]


def summary_of(scores: Sequence[float], values: np.ndarray) -> Summary:
    """Summary of a set of scores with value rows, straight from its definition.

    m = max s_i;  l = sum_i exp(s_i - m);  o~ = sum_i exp(s_i - m) v_i.
    The empty set (or a set of -inf scores) is the identity (-inf, 0, 0).
    """
    values = np.asarray(values, dtype=np.float64)
    dv = values.shape[1] if values.ndim == 2 else 0
    s = np.asarray(scores, dtype=np.float64)
    if s.size == 0 or np.all(np.isneginf(s)):
        return (NEG_INF, 0.0, np.zeros(dv))
    m = float(np.max(s))
    w = np.exp(s - m)
    return (m, float(np.sum(w)), w @ values)


def merge(a: Summary, b: Summary) -> Summary:
    """The merge of two summaries: bring both to the larger max, then add.

    m = max(m_a, m_b);  l = l_a e^{m_a - m} + l_b e^{m_b - m};
    o~ = o~_a e^{m_a - m} + o~_b e^{m_b - m}.
    A side whose max is -inf is the identity and gets weight 0 (this avoids
    e^{-inf - (-inf)} = NaN, [P3] property 2).
    """
    ma, la, oa = a
    mb, lb, ob = b
    m = max(ma, mb)
    if m == NEG_INF:
        return (NEG_INF, 0.0, np.zeros_like(np.asarray(oa, dtype=np.float64)))
    wa = 0.0 if ma == NEG_INF else math.exp(ma - m)
    wb = 0.0 if mb == NEG_INF else math.exp(mb - m)
    return (m, la * wa + lb * wb, np.asarray(oa) * wa + np.asarray(ob) * wb)


def merge_all(parts: Sequence[Summary]) -> Summary:
    """Left-to-right merge of a list of summaries (identity for an empty list)."""
    if not parts:
        raise ValueError("merge_all needs at least one summary (it fixes d_v)")
    acc = parts[0]
    for p in parts[1:]:
        acc = merge(acc, p)
    return acc


def finalize(p: Summary) -> Tuple[np.ndarray, float]:
    """(o, lse) from a summary: o = o~ / l, lse = m + log l.

    l = 0 (the identity, a fully masked row) gives o = 0 and lse = -inf.
    [P3] "From weights to outputs" (one division at the end; lse = m_n + log l_n).
    """
    m, l, o = p
    if l == 0.0:
        return np.zeros_like(np.asarray(o, dtype=np.float64)), NEG_INF
    return np.asarray(o, dtype=np.float64) / l, m + math.log(l)


def lse_merge_ref(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Merge of normalised partial results (o_s, lse_s) in log-sum-exp form.

    lse = log sum_s e^{lse_s} (computed as max + log sum e^{lse_s - max});
    o = sum_s e^{lse_s - lse} o_s, a convex combination.  A part with
    lse_s = -inf has weight 0; if every part is -inf, o = 0 and lse = -inf.

    o_parts: [S, rows, d]; lse_parts: [S, rows].  Returns (o [rows, d], lse [rows]).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = np.max(lse_parts, axis=0)
    ref = np.where(np.isneginf(mx), 0.0, mx)
    w = np.exp(lse_parts - ref[None, :])  # -inf parts -> 0
    tot = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, ref + np.log(np.where(tot > 0, tot, 1.0)), NEG_INF)
        wn = np.where(tot[None, :] > 0, w / np.where(tot > 0, tot, 1.0)[None, :], 0.0)
    o = np.einsum("sr,srd->rd", wn, o_parts)
    return o, lse


# ---------------------------------------------------------------------------
# Attention.
# Plain definition: [P1] "naive_attention" in "How does the online softmax
# recurrence work?"; [P3] "Blocks, the bridge to FlashAttention" (S = Q K^T
# scaled); masks: [P2] "Masks belong inside the tiled loop".
# ---------------------------------------------------------------------------


def visible_keys(i: int, nq: int, nk: int, causal: bool, key_len: int) -> int:
    """Number of keys query row i may attend to (keys 0 .. count-1)."""
    lim = min(max(int(key_len), 0), nk)
    if causal:
        lim = min(lim, i + 1 + (nk - nq))
    return max(lim, 0)


def attention_ref(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  causal: bool = False, key_len=None, rows=None,
                  block_rows: int = 512) -> Tuple[np.ndarray, np.ndarray]:
    """Exact softmax attention in float64 by its plain definition.

    q: [B, H, Nq, d], k, v: [B, H, Nk, d].  For every (b, h) and query row i:
        s_ij = scale * (q_i . k_j)                 for every key j
        s_ij = -inf   if j >= key_len[b] or (causal and j > i + Nk - Nq)
        p_i  = safe softmax of s_i (three passes); a fully masked row gives 0
        o_i  = p_i V;   lse_i = log sum_j exp(s_ij)  (-inf for a masked row)
    ``rows`` optionally restricts the query rows computed (an index array into
    Nq, the same for every (b, h)); outputs then have that many rows.
    Returns (o [B, H, R, d] float64, lse [B, H, R] float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if key_len is None:
        key_len = [Nk] * B
    key_len = [int(x) for x in np.asarray(key_len).reshape(-1)]
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    R = rows.size
    o = np.zeros((B, H, R, v.shape[3]))
    lse = np.full((B, H, R), NEG_INF)
    kidx = np.arange(Nk)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, R, block_rows):
                ri = rows[r0:r0 + block_rows]
                s = scale * (q[b, h, ri, :] @ k[b, h].T)             # [r, Nk]
                lim = np.minimum(max(min(key_len[b], Nk), 0), Nk)
                vis = kidx[None, :] < lim
                if causal:
                    vis = vis & (kidx[None, :] <= (ri[:, None] + (Nk - Nq)))
                s = np.where(vis, s, NEG_INF)
                m = np.max(s, axis=1, keepdims=True)                 # pass 1
                ref = np.where(np.isneginf(m), 0.0, m)
                e = np.exp(s - ref)                                  # pass 2
                l = np.sum(e, axis=1, keepdims=True)
                safe_l = np.where(l > 0, l, 1.0)
                p = np.where(l > 0, e / safe_l, 0.0)                 # pass 3
                o[b, h, r0:r0 + ri.size] = p @ v[b, h]
                with np.errstate(divide="ignore"):
                    lse[b, h, r0:r0 + ri.size] = np.where(
                        l[:, 0] > 0, ref[:, 0] + np.log(safe_l[:, 0]), NEG_INF)
    return o, lse


def attention_bwd_ref(q, k, v, o, lse, do, scale: float, causal: bool = False,
                      key_len=None, parts: bool = False):
    """Gradients of softmax attention in float64, from the forward's o and lse.

    [P3] "From weights to outputs": the log-sum-exp is all the backward pass
    needs to rebuild the weights, p_ij = exp(s_ij - lse_i).  With the masks of
    ``attention_ref`` (p = 0 where masked, and for a row with lse = -inf):
        dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
        dS = P * (dP - D_i),  dQ = scale dS K,  dK = scale dS^T Q.
    These are the derivatives of sum(dO * O) for O = softmax(s) V; the pins
    check them against finite differences of ``attention_ref``.
    Returns (dq, dk, dv) float64; with ``parts`` also, per (b, h), the
    arrays (|P|^T |dO|, scale |dS| |K|, scale |dS|^T |Q|) that bound the
    rounding of the terms (used for the GPU tolerance).
    """
    q, k, v, o, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, o, do))
    lse = np.asarray(lse, dtype=np.float64)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if key_len is None:
        key_len = [Nk] * B
    key_len = [int(x) for x in np.asarray(key_len).reshape(-1)]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    bounds = (np.zeros_like(v), np.zeros_like(q), np.zeros_like(k)) if parts else None
    kidx, qidx = np.arange(Nk), np.arange(Nq)
    for b in range(B):
        lim = min(max(key_len[b], 0), Nk)
        vis = np.broadcast_to(kidx[None, :] < lim, (Nq, Nk))
        if causal:
            vis = vis & (kidx[None, :] <= qidx[:, None] + (Nk - Nq))
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)
            live = np.isfinite(lse[b, h])[:, None] & vis
            with np.errstate(invalid="ignore", over="ignore"):
                p = np.where(live, np.exp(np.where(live, s, 0.0) - np.where(
                    np.isfinite(lse[b, h]), lse[b, h], 0.0)[:, None]), 0.0)
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            D = np.sum(do[b, h] * o[b, h], axis=1)
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
            if parts:
                bounds[0][b, h] = np.abs(p).T @ np.abs(do[b, h])
                bounds[1][b, h] = scale * (np.abs(ds) @ np.abs(k[b, h]))
                bounds[2][b, h] = scale * (np.abs(ds).T @ np.abs(q[b, h]))
    if parts:
        return dq, dk, dv, bounds
    return dq, dk, dv


def attention_bruteforce(q, k, v, scale, causal=False, key_len=None):
    """Attention by explicit loops and exactly rounded sums (tiny inputs only).

    Independent of NumPy's matmul and reductions: every dot product and every
    sum goes through math.fsum.  Same shapes and masking rules as
    ``attention_ref``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Nq, d = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    if key_len is None:
        key_len = [Nk] * B
    o = np.zeros((B, H, Nq, dv))
    lse = np.full((B, H, Nq), NEG_INF)
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                n = visible_keys(i, Nq, Nk, causal, int(key_len[b]))
                if n == 0:
                    continue
                s = [scale * math.fsum(q[b, h, i, t] * k[b, h, j, t] for t in range(d))
                     for j in range(n)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                l = math.fsum(e)
                for c in range(dv):
                    o[b, h, i, c] = math.fsum(e[j] * v[b, h, j, c] for j in range(n)) / l
                lse[b, h, i] = m + math.log(l)
    return o, lse


def online_attention_single(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                            scale: float = 1.0, block: int = 64) -> Tuple[np.ndarray, float]:
    """One query, keys and values streamed in blocks, with the online recurrence.

    [P1] "How does the online softmax recurrence work?": keep running max m,
    running sum l and running unnormalised output O; for each block of keys
    take the block scores, the new max, the shrink factor exp(m - m_new) for
    the old state, the block weights exp(s - m_new); update l and O; divide
    once at the end.  Also returns lse = m + log l ([P3] "From weights to
    outputs").  q: [d], k, v: [N, d].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m, l = NEG_INF, 0.0
    acc = np.zeros(v.shape[1])
    for start in range(0, k.shape[0], block):
        s = scale * (k[start:start + block] @ q)
        m_new = max(m, float(np.max(s)))
        shrink = 0.0 if m == NEG_INF else math.exp(m - m_new)
        w = np.exp(s - m_new)
        l = shrink * l + float(np.sum(w))
        acc = shrink * acc + w @ v[start:start + block]
        m = m_new
    return acc / l, m + math.log(l)


def online_attention_single_normalised(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                                       scale: float = 1.0,
                                       block: int = 64) -> Tuple[np.ndarray, float]:
    """The same stream, keeping the output normalised after every block.

    [P3] "From weights to outputs", the second way to write it (the form of
    the original FlashAttention): with o = O~ / l held instead of O~, a block
    step is o_new = (l e^{m - m_new} o + sum_j e^{s_j - m_new} v_j) / l_new,
    one division per step instead of one at the end.  Both forms are exact;
    the pages call the per-step division wasted work.  Returns (o, lse).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m, l = NEG_INF, 0.0
    o = np.zeros(v.shape[1])
    for start in range(0, k.shape[0], block):
        s = scale * (k[start:start + block] @ q)
        m_new = max(m, float(np.max(s)))
        shrink = 0.0 if m == NEG_INF else math.exp(m - m_new)
        w = np.exp(s - m_new)
        l_new = shrink * l + float(np.sum(w))
        o = (shrink * l * o + w @ v[start:start + block]) / l_new
        m, l = m_new, l_new
    return o, m + math.log(l)


# ---------------------------------------------------------------------------
# Helpers used only by the pin tests.
# ---------------------------------------------------------------------------


def set_partitions(items: Sequence[int]):
    """All set partitions of ``items`` (Bell-number many; small inputs only)."""
    items = list(items)
    if not items:
        yield []
        return
    first, rest = items[0], items[1:]
    for part in set_partitions(rest):
        for i in range(len(part)):
            yield part[:i] + [[first] + part[i]] + part[i + 1:]
        yield [[first]] + part


def all_orders_and_groupings(n: int):
    """Every set partition of range(n), each block list in every order."""
    for part in set_partitions(range(n)):
        for perm in itertools.permutations(part):
            yield list(perm)
