"""The seeded input generators: shapes, value recipe and determinism (CPU)."""
import numpy as np
import torch

import workloads as W


def test_softmax_logits_recipe():
    x = W.softmax_logits(seed=2, rows=64, cols=1000)
    assert x.shape == (64, 1000) and x.dtype == torch.float32
    assert int((x == 40.0).sum()) == round(0.01 * 64 * 1000)
    rest = x[x != 40.0]
    assert abs(float(rest.std()) - 2.0) < 0.1          # variance 4
    assert torch.equal(x, W.softmax_logits(seed=2, rows=64, cols=1000))


def test_attention_recipe():
    c = W.attention(4, 3, 2, 40, 40, 16, True, (10, 40))
    assert c.q.dtype == torch.bfloat16 and c.q.shape == (3, 2, 40, 16)
    assert c.key_len.dtype == torch.int32 and c.key_len.shape == (3,)
    assert int(c.key_len.min()) >= 10 and int(c.key_len.max()) <= 40
    assert abs(c.scale - 0.25) < 1e-15
    c2 = W.attention(4, 3, 2, 40, 40, 16, True, (10, 40))
    assert torch.equal(c.k, c2.k) and torch.equal(c.key_len, c2.key_len)


def test_decode_recipe_small():
    c = W.decode(seed=5, B=3, H=2, Nk=256, d=16, len_range=(10, 256), num_splits=4,
                 spike_frac=0.01, keep_host=(1,))
    assert c.k.shape == (3, 2, 256, 16) and c.q.shape == (3, 2, 1, 16)
    for b in range(3):
        n = int(c.key_len[b])
        assert torch.all(c.k[b, :, n:] == 0) and torch.all(c.v[b, :, n:] == 0)
    assert torch.equal(c.meta_host[1][0], c.k[1])
    big = (c.k.float().abs() > 6.0).any(-1).sum()
    assert int(big) >= 1                              # some keys were scaled by 8
