"""Attention backward on the GPU against the float64 oracle.

Inputs: q, k, v, dO bf16; O (rounded to bf16) and lse (fp32) from the
oracle's own forward, so nothing fed to either side comes from the CUDA path.
Bar, element by element, derived from the kernel's arithmetic: P and dS are
rounded to bf16 (unit roundoff 2^-8) before the products that use them, and
the outputs are stored in bf16 (another 2^-8 relative), so
  |dV - dV_ref| <= 2^-8 (|P|^T |dO|) + 2^-8 |dV_ref| + 1e-4,
  |dQ - dQ_ref| <= 2^-8 scale (|dS| |K|) + 2^-8 |dQ_ref| + 1e-4,
  |dK - dK_ref| <= 2^-8 scale (|dS|^T |Q|) + 2^-8 |dK_ref| + 1e-4
(the first term is the P / dS rounding with every error aligned; the fp32
accumulation and exp2 error are below the absolute term).
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

_DO = 7  # tensor id of dO within a case's seed


def make_case(seed, B, H, Nq, Nk, causal, len_range=None, key_len=None, d=128):
    c = W.attention(seed, B, H, Nq, Nk, d, causal, len_range)
    if key_len is not None:
        c.key_len = torch.tensor(key_len, dtype=torch.int32)
    do = W.to_bf16(W.normal_bhnd(seed, _DO, B, H, Nq, d))
    kl = c.key_len.numpy() if c.key_len is not None else None
    o64, lse64 = oracle.attention_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), c.scale,
                                      causal, kl)
    o = torch.from_numpy(o64).to(torch.bfloat16)
    lse = torch.from_numpy(lse64).to(torch.float32)
    return c, do, o, lse


def run_gpu(c, do, o, lse):
    kl = c.key_len.cuda() if c.key_len is not None else None
    g = osm.attn_bwd(c.q.cuda(), c.k.cuda(), c.v.cuda(), o.cuda(), lse.cuda(), do.cuda(),
                     c.scale, c.causal, kl)
    assert osm.device_status() == 0
    return g


def check(c, do, o, lse, got):
    kl = c.key_len.numpy() if c.key_len is not None else None
    dq, dk, dv, (bv, bq, bk) = oracle.attention_bwd_ref(
        W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), W.as_f64(o), W.as_f64(lse), W.as_f64(do),
        c.scale, c.causal, kl, parts=True)
    for name, g, ref, bound in (("dq", got[0], dq, bq), ("dk", got[1], dk, bk),
                                ("dv", got[2], dv, bv)):
        g = W.as_f64(g)
        assert np.all(np.isfinite(g)), name
        excess = np.abs(g - ref) - (2.0 ** -8 * bound + 2.0 ** -8 * np.abs(ref) + 1e-4)
        assert float(excess.max()) <= 0, f"{name}: worst excess {excess.max()}"


SHAPES = [(1, 1, 1, 1), (1, 1, 63, 63), (1, 2, 64, 64), (2, 1, 127, 129), (1, 1, 129, 127),
          (1, 2, 300, 300), (1, 1, 257, 1000), (1, 1, 1000, 257), (2, 2, 513, 513)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(cuda_ok, shape, causal):
    B, H, Nq, Nk = shape
    c, do, o, lse = make_case(sum(shape) + 200 * causal, B, H, Nq, Nk, causal,
                              (max(1, Nk // 3), Nk))
    check(c, do, o, lse, run_gpu(c, do, o, lse))


@pytest.mark.parametrize("causal", [False, True])
def test_key_len_edges(cuda_ok, causal):
    """key_len 0 (every gradient 0), 1, N-1, N; keys past key_len get dK = dV = 0."""
    N = 300
    c, do, o, lse = make_case(31 + causal, 4, 2, N, N, causal, key_len=[0, 1, N - 1, N])
    got = run_gpu(c, do, o, lse)
    check(c, do, o, lse, got)
    for g in got:
        assert torch.all(g[0] == 0)
    assert torch.all(got[1][1, :, 1:] == 0) and torch.all(got[2][1, :, 1:] == 0)


def test_more_queries_than_keys_causal(cuda_ok):
    """Bottom-right causal with Nq > Nk: the first Nq - Nk rows see no key."""
    c, do, o, lse = make_case(33, 1, 2, 400, 150, True)
    got = run_gpu(c, do, o, lse)
    check(c, do, o, lse, got)
    assert torch.all(got[0][:, :, :250] == 0)


def test_medium_causal_padded(cuda_ok):
    c, do, o, lse = make_case(34, 2, 4, 2048, 2048, True, (1024, 2048))
    check(c, do, o, lse, run_gpu(c, do, o, lse))


def test_deterministic(cuda_ok):
    c, do, o, lse = make_case(35, 1, 2, 700, 700, True, (300, 700))
    a = run_gpu(c, do, o, lse)
    b = run_gpu(c, do, o, lse)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_full_size_causal_padded_sampled_heads(cuda_ok):
    """The forward benchmark's shape (B8 H32 N8192 d128, causal, key_len
    U[4096, 8192]) in the launch configuration the profiles time: every
    gradient of head 0 of the batches with the shortest and the longest key
    length against the oracle.  The other heads get O = 0 and lse = 0 (finite
    inputs; their gradients are not checked)."""
    B, H, N = 8, 32, 8192
    c = W.attention(4, B, H, N, N, 128, True, (4096, 8192))
    do = W.to_bf16(W.normal_bhnd(4, _DO, B, H, N, 128))
    lens = c.key_len.numpy()
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens))})
    o = torch.zeros_like(c.q)
    lse = torch.zeros((B, H, N), dtype=torch.float32)
    for b in picks:
        o64, l64 = oracle.attention_ref(W.as_f64(c.q[b:b + 1, :1]), W.as_f64(c.k[b:b + 1, :1]),
                                        W.as_f64(c.v[b:b + 1, :1]), c.scale, True, lens[b:b + 1])
        o[b, 0] = torch.from_numpy(o64[0, 0]).to(torch.bfloat16)
        lse[b, 0] = torch.from_numpy(l64[0, 0]).to(torch.float32)
    got = run_gpu(c, do, o, lse)
    for b in picks:
        sub = W.AttnCase(c.q[b:b + 1, :1], c.k[b:b + 1, :1], c.v[b:b + 1, :1], c.scale, True,
                         c.key_len[b:b + 1])
        check(sub, do[b:b + 1, :1], o[b:b + 1, :1], lse[b:b + 1, :1],
              tuple(g[b:b + 1, :1] for g in got))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 65, 65), (2, 1, 127, 129), (1, 2, 300, 300),
                                   (1, 1, 1000, 257), (2, 2, 513, 513)])
def test_head_dim_64(cuda_ok, shape, causal):
    B, H, Nq, Nk = shape
    c, do, o, lse = make_case(sum(shape) + 400 + 9 * causal, B, H, Nq, Nk, causal,
                              (max(1, Nk // 3), Nk), d=64)
    check(c, do, o, lse, run_gpu(c, do, o, lse))


def test_head_dim_64_key_len_edges(cuda_ok):
    N = 300
    c, do, o, lse = make_case(36, 4, 2, N, N, True, key_len=[0, 1, N - 1, N], d=64)
    got = run_gpu(c, do, o, lse)
    check(c, do, o, lse, got)
    for g in got:
        assert torch.all(g[0] == 0)
