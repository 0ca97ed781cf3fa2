"""Run every operation of a library built with OSM_CHECKED on small and edge
shapes: no index check may fire (osm_device_status reports OSM_ERR_INDEX
when one does) and every result must match the float64 oracle at the usual
bars.  Usage: python checked_cases.py <path to libosm_checked.so>.  Run in a
process of its own, so that no other build of the library is loaded."""
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import exact_tiled_attention_osm_gb300 as osm  # noqa: E402

osm.load_library(sys.argv[1])

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from bars import check_attention  # noqa: E402


def clean(what):
    w = osm.device_status()
    assert w == 0, f"{what}: device status word {w:#x}"


def attention_cases():
    n = 0
    for d in (64, 128):
        for causal in (False, True):
            for (B, H, Nq, Nk) in ((1, 1, 1, 1), (2, 1, 127, 129), (1, 2, 300, 300), (1, 1, 257, 1000),
                                   (2, 1, 400, 150)):
                c = W.attention(Nq + Nk + d + causal, B, H, Nq, Nk, d, causal, (max(1, Nk // 3), Nk))
                kl = c.key_len.cuda()
                ro, rl = oracle.attention_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), c.scale,
                                              causal, c.key_len.numpy())
                for kw in ({}, {"score_bound": 4.0}, {"normalised": True}):
                    o, lse = osm.attn_fwd(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.scale, causal, kl, **kw)
                    clean(f"attn_fwd d{d} causal={causal} {(B, H, Nq, Nk)} {kw}")
                    check_attention(W.as_f64(o), W.as_f64(lse), ro, rl)
                    n += 1
    c = W.attention(7, 4, 2, 300, 300, 128, True, None)
    c.key_len = torch.tensor([0, 1, 299, 300], dtype=torch.int32)
    o, lse = osm.attn_fwd(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.scale, True, c.key_len.cuda())
    clean("attn_fwd key_len edges")
    check_attention(W.as_f64(o), W.as_f64(lse),
                    *oracle.attention_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), c.scale, True,
                                          c.key_len.numpy()))
    return n + 1


def backward_cases():
    n = 0
    for d in (64, 128):
        c = W.attention(40 + d, 2, 2, 300, 300, d, True, (100, 300))
        kl = c.key_len.cuda()
        ro, rl = oracle.attention_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), c.scale, True,
                                      c.key_len.numpy())
        o = torch.from_numpy(ro).to(torch.bfloat16)
        lse = torch.from_numpy(rl).to(torch.float32)
        do = W.to_bf16(W.normal_bhnd(41 + d, 7, 2, 2, 300, d))
        grads = osm.attn_bwd(c.q.cuda(), c.k.cuda(), c.v.cuda(), o.cuda(), lse.cuda(), do.cuda(),
                             c.scale, True, kl)
        clean(f"attn_bwd d{d}")
        refs = oracle.attention_bwd_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), W.as_f64(o),
                                        W.as_f64(lse), W.as_f64(do), c.scale, True,
                                        c.key_len.numpy(), parts=True)
        for g, ref, bound in zip(grads, refs[:3], (refs[3][1], refs[3][2], refs[3][0])):
            excess = np.abs(W.as_f64(g) - ref) - (2.0 ** -8 * bound + 2.0 ** -8 * np.abs(ref) + 1e-4)
            assert excess.max() <= 0, f"backward d{d} excess {excess.max()}"
        n += 1
    return n


def decode_cases():
    n = 0
    for dtype in (torch.bfloat16, torch.float32):
        for d in (64, 128):
            for splits in (1, 3, 16):
                case = W.decode(seed=60 + d + splits, B=3, H=2, Nk=700, d=d, len_range=(1, 700),
                                num_splits=splits)
                kl = case.key_len.clone()
                kl[0] = 0
                q, k, v = (t.to(dtype) for t in (case.q, case.k, case.v))
                o, lse = osm.attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), case.scale, kl.cuda(),
                                                 splits)
                clean(f"decode {dtype} d{d} splits{splits}")
                ro, rl = oracle.attention_ref(W.as_f64(q), W.as_f64(k), W.as_f64(v), case.scale, False,
                                              kl.numpy())
                if dtype == torch.float32:
                    assert np.max(np.abs(W.as_f64(o)[:, :, 0] - ro[:, :, 0])) <= 1e-5
                else:
                    check_attention(W.as_f64(o)[:, :, 0], W.as_f64(lse), ro[:, :, 0], rl[:, :, 0])
                n += 1
    # append: extend an empty state by all keys
    case = W.decode(seed=70, B=2, H=2, Nk=500, d=128, len_range=(100, 500), num_splits=5)
    state = osm.decode_state(2, 2, 128, torch.device("cuda"))
    o, lse = osm.attn_decode_append(case.q.cuda(), case.k.cuda(), case.v.cuda(), state, None,
                                    case.key_len.cuda(), case.scale, 5)
    clean("decode append")
    ro, rl = oracle.attention_ref(W.as_f64(case.q), W.as_f64(case.k), W.as_f64(case.v), case.scale,
                                  False, case.key_len.numpy())
    check_attention(W.as_f64(o)[:, :, 0], W.as_f64(lse), ro[:, :, 0], rl[:, :, 0])
    # LSE-form merge
    rng = np.random.default_rng(3)
    op = rng.standard_normal((5, 200, 128)).astype(np.float32)
    lp = (rng.standard_normal((5, 200)) * 4).astype(np.float32)
    lp[1, :30] = -np.inf
    o, lse = osm.lse_merge(torch.from_numpy(op).cuda(), torch.from_numpy(lp).cuda(), torch.float32)
    clean("lse_merge")
    ro, rl = oracle.lse_merge_ref(op.astype(np.float64), lp.astype(np.float64))
    assert np.max(np.abs(W.as_f64(o) - ro)) <= 1e-5
    return n + 2


def softmax_cases():
    n = 0
    for rows, cols in ((1, 1), (3, 4), (5, 7), (2, 4100), (3, 32768), (2, 131076), (300, 96)):
        x = W.softmax_logits(seed=rows + cols, rows=rows, cols=cols)
        y = osm.softmax_rows(x.cuda())
        clean(f"softmax {rows}x{cols}")
        ref = oracle.softmax_rows_ref(W.as_f64(x))
        assert np.max(np.abs(W.as_f64(y) - ref) / np.maximum(np.abs(ref), 1e-30)) <= 1e-5
        for k in (1, 8):
            if k > cols:
                continue
            idx, prob = osm.softmax_topk(x.cuda(), k)
            clean(f"softmax_topk {rows}x{cols} k{k}")
            ri, rp = oracle.softmax_topk_ref(W.as_f64(x), k)
            assert np.array_equal(idx.cpu().numpy().astype(np.int64), ri)
        n += 1
    return n


if __name__ == "__main__":
    torch.cuda.set_device(0)
    counts = {"attention": attention_cases(), "backward": backward_cases(),
              "decode": decode_cases(), "softmax": softmax_cases()}
    print("checked build clean:", counts)
