"""Split-KV decode and the log-sum-exp merge on the GPU against the float64 oracle.

Bars: FP32 inputs (single-query workload): O and LSE within 1e-5 absolute.
BF16 inputs: the bars of ``bars.py`` -- O within 1e-2 on every element of
the full-size workload, elsewhere within 1e-2 + 2^-8 |O_ref| (the value plus
the bf16 output's own rounding); LSE within 1e-3.  Workspace partials: every non-empty split has
1 <= l <= (its key count) and m equal to the split's maximum score.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import check_attention, o_bar, record

pytestmark = pytest.mark.gpu


def ref_decode(q, k, v, scale, key_len):
    return oracle.attention_ref(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False,
                                None if key_len is None else key_len.cpu().numpy())


def check_bf16(o, lse, ro, rl, plain=False):
    return check_attention(W.as_f64(o)[:, :, 0], W.as_f64(lse), ro[:, :, 0], rl[:, :, 0], plain)


@pytest.mark.parametrize("splits", [1, 64])
def test_single_query_fp32(cuda_ok, splits):
    """q (64,), K, V (4096, 64) fp32 N(0,1), scale 1, against softmax-then-PV."""
    q, k, v, scale = W.single_query(1)
    o, lse = osm.attn_decode_splitkv(q.view(1, 1, 1, 64).cuda(), k.view(1, 1, 4096, 64).cuda(),
                                     v.view(1, 1, 4096, 64).cuda(), scale, None, splits)
    assert osm.device_status() == 0
    ro, rl = oracle.attention_ref(W.as_f64(q)[None, None, None], W.as_f64(k)[None, None],
                                  W.as_f64(v)[None, None], scale)
    assert float(np.max(np.abs(W.as_f64(o).reshape(-1) - ro.reshape(-1)))) <= 1e-5
    assert abs(float(lse.item()) - float(rl.item())) <= 1e-5
    # and against the pages' blockwise single-query loop (block 64)
    oo, ll = oracle.online_attention_single(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, 64)
    assert float(np.max(np.abs(W.as_f64(o).reshape(-1) - oo))) <= 1e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 16, 256])
def test_small_ragged(cuda_ok, dtype, d, splits):
    B, H, Nk = 4, 3, 1000
    case = W.decode(seed=30 + d + splits, B=B, H=H, Nk=Nk, d=d, len_range=(1, Nk),
                    num_splits=splits)
    kl = case.key_len.clone()
    kl[0] = 0          # no keys at all
    kl[1] = 1          # a single key
    q, k, v = (t.to(dtype) for t in (case.q, case.k, case.v))
    o, lse = osm.attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), case.scale, kl.cuda(), splits)
    assert osm.device_status() == 0
    ro, rl = ref_decode(q, k, v, case.scale, kl)
    if dtype == torch.float32:
        assert float(np.max(np.abs(W.as_f64(o)[:, :, 0] - ro[:, :, 0]))) <= 1e-5
        fin = np.isfinite(rl[:, :, 0])
        assert np.array_equal(np.isneginf(W.as_f64(lse)), ~fin)
        assert float(np.max(np.abs(W.as_f64(lse)[fin] - rl[:, :, 0][fin]))) <= 1e-5
    else:
        check_bf16(o, lse, ro, rl)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_largest_grid(cuda_ok):
    """B = 65535 (the largest batch the decode grid takes), one head, short
    ragged caches, 3 splits: every row against the oracle."""
    B, H, Nk, d = 65535, 1, 40, 64
    g = torch.Generator().manual_seed(36)  # one draw for all rows (fast at this batch)
    q = torch.randn(B, H, 1, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Nk, d, generator=g).to(torch.bfloat16)
    kl = torch.randint(0, Nk + 1, (B,), generator=g, dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    o, lse = osm.attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), scale, kl.cuda(), 3)
    assert osm.device_status() == 0
    ro, rl = ref_decode(q, k, v, scale, kl)
    check_bf16(o, lse, ro, rl)


def test_partials_in_workspace(cuda_ok):
    B, H, Nk, d, S = 3, 2, 2000, 128, 16
    case = W.decode(seed=40, B=B, H=H, Nk=Nk, d=d, len_range=(5, Nk), num_splits=S)
    ws = torch.empty(osm.decode_workspace_bytes(B, H, d, S), dtype=torch.uint8, device="cuda")
    osm.attn_decode_splitkv(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale,
                            case.key_len.cuda(), S, workspace=ws)
    assert osm.device_status() == 0
    m, l, ot = (W.as_f64(t) for t in osm.decode_partials(ws, B, H, d, S))
    q64, k64, v64 = W.as_f64(case.q), W.as_f64(case.k), W.as_f64(case.v)
    parts = [[] for _ in range(B * H)]
    for b in range(B):
        L = int(case.key_len[b])
        c = -(-L // S)
        for h in range(H):
            r = b * H + h
            for s in range(S):
                lo, hi = min(L, s * c), min(L, s * c + c)
                if lo >= hi:
                    assert m[s, r] == -math.inf and l[s, r] == 0 and np.all(ot[s, r] == 0)
                    parts[r].append((-math.inf, 0.0, np.zeros(d)))
                    continue
                sc = case.scale * (k64[b, h, lo:hi] @ q64[b, h, 0])
                assert 1.0 - 1e-5 <= l[s, r] <= (hi - lo) * (1 + 1e-5)
                assert abs(m[s, r] - sc.max()) <= 1e-4 * max(1.0, abs(sc.max()))
                want = oracle.summary_of(sc, v64[b, h, lo:hi])
                assert abs(l[s, r] - want[1]) <= 1e-3 * want[1]
                assert np.max(np.abs(ot[s, r] - want[2])) <= 1e-2 * max(1.0, want[1])
                parts[r].append((m[s, r], l[s, r], ot[s, r]))
    # merging the stored partials on the CPU gives the whole row
    ro, rl = ref_decode(case.q, case.k, case.v, case.scale, case.key_len)
    for r in range(B * H):
        o_m, lse_m = oracle.finalize(oracle.merge_all(parts[r]))
        b, h = divmod(r, H)
        assert np.max(np.abs(o_m - ro[b, h, 0])) <= 1e-3
        assert abs(lse_m - rl[b, h, 0]) <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge(cuda_ok, d, out_dtype):
    rng = np.random.default_rng(d)
    S, rows = 7, 300
    o_parts = rng.standard_normal((S, rows, d)).astype(np.float32)
    lse_parts = (rng.standard_normal((S, rows)) * 5).astype(np.float32)
    lse_parts[2, :50] = -np.inf           # empty pieces
    lse_parts[:, 60] = -np.inf            # a row with no piece at all
    o, lse = osm.lse_merge(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda(),
                           out_dtype)
    ro, rl = oracle.lse_merge_ref(o_parts.astype(np.float64), lse_parts.astype(np.float64))
    bar = 1e-5 if out_dtype == torch.float32 else o_bar(ro)
    assert np.all(np.abs(W.as_f64(o) - ro) <= bar)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(W.as_f64(lse)), ~fin)
    assert float(np.max(np.abs(W.as_f64(lse)[fin] - rl[fin]))) <= 1e-5
    assert torch.all(o[60] == 0)


def test_deterministic(cuda_ok):
    case = W.decode(seed=41, B=2, H=4, Nk=5000, d=128, len_range=(100, 5000), num_splits=16)
    a = osm.attn_decode_splitkv(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale,
                                case.key_len.cuda(), 16)
    b = osm.attn_decode_splitkv(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale,
                                case.key_len.cuda(), 16)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_full_size_decode(cuda_ok):
    """B64 H32 Nk32768 d128 bf16, 0.1% of keys x8, key_len ~ U[1024, 32768], 16
    splits: every head of four batch entries (incl. the shortest and longest)."""
    lens = W.key_lengths(5, 64, 1024, 32768)
    keep = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 0, 63})
    case = W.decode(seed=5, device="cuda", keep_host=keep)
    o, lse = osm.attn_decode_splitkv(case.q, case.k, case.v, case.scale, case.key_len,
                                     case.num_splits)
    assert osm.device_status() == 0
    eo = el = 0.0
    for b in keep:
        kb, vb = case.meta_host[b]
        ro, rl = oracle.attention_ref(W.as_f64(case.q[b:b + 1].cpu()), W.as_f64(kb[None]),
                                      W.as_f64(vb[None]), case.scale, False, [int(lens[b])])
        e = check_bf16(o[b:b + 1], lse[b:b + 1], ro, rl, plain=True)
        eo, el = max(eo, e[0]), max(el, e[1])
    record("decode B64 H32 Nk32768 d128 16 splits (every head of 4 batch entries)",
           o_err=eo, lse_err=el)
    assert torch.all(torch.isfinite(o)) and torch.all(torch.isfinite(lse))


def test_very_long_cache(cuda_ok):
    """One query per head against 262144 keys (16 splits of 16384 keys), key
    lengths 262144 and 100001."""
    B, H, Nk = 2, 2, 262144
    case = W.decode(seed=43, B=B, H=H, Nk=Nk, d=128, len_range=(Nk, Nk), num_splits=16)
    kl = torch.tensor([Nk, 100001], dtype=torch.int32)
    o, lse = osm.attn_decode_splitkv(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale,
                                     kl.cuda(), 16)
    assert osm.device_status() == 0
    check_bf16(o, lse, *ref_decode(case.q, case.k, case.v, case.scale, kl))
