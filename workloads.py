"""Seeded synthetic inputs for the five workloads of exact online-softmax attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Tests, the smoke check and the benchmark take their
inputs from here, and the same CPU values (upcast to float64) go to the oracle.

Random streams: NumPy PCG64 seeded with SeedSequence([seed, tensor_id, part]),
so every tensor (and every part of a large tensor) has its own stream and the
values do not depend on thread count or on the order parts are generated in.
BF16 inputs are drawn in float32 and rounded to bfloat16 (round to nearest
even, by torch's conversion); that rounded tensor is what both sides see.

Workloads (names used by the tests and the benchmark):
  single_query   q (64,), K, V (4096, 64) fp32 N(0,1), scale 1, no mask
  softmax_rows   x (4096, 32768) fp32 = 2 * N(0,1) (variance 4), plus
                 round(0.01 * rows * cols) distinct flat positions set to 40.0
  attn           Q, K, V (4, 16, 4096, 128) bf16 N(0,1), scale 1/sqrt(128)
  attn_causal    Q, K, V (8, 32, 8192, 128) bf16 N(0,1), causal, valid key
                 length per batch uniform on [4096, 8192]
  decode         q (64, 32, 1, 128), K, V (64, 32, 32768, 128) bf16 N(0,1);
                 round(0.001 * B * H * Nk) distinct key rows of K scaled by 8
                 (in fp32, before bf16 rounding); valid length per batch
                 uniform on [1024, 32768]; keys past the valid length are 0
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

# tensor ids inside one workload's seed
_Q, _K, _V, _X, _LEN, _SPIKE = 1, 2, 3, 4, 5, 6


def _gen(seed: int, tensor_id: int, part: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, part])))


def normal_f32(seed: int, tensor_id: int, shape: Sequence[int], part: int = 0,
               sigma: float = 1.0) -> np.ndarray:
    x = _gen(seed, tensor_id, part).standard_normal(size=tuple(shape), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def _threads() -> int:
    return max(1, min(16, len(os.sched_getaffinity(0))))


def normal_bhnd(seed: int, tensor_id: int, B: int, H: int, N: int, d: int,
                lengths: Optional[Sequence[int]] = None) -> np.ndarray:
    """fp32 [B, H, N, d]; part (b, h) has its own stream; rows >= lengths[b] are 0."""
    out = np.zeros((B, H, N, d), dtype=np.float32)

    def work(bh):
        b, h = divmod(bh, H)
        n = N if lengths is None else int(lengths[b])
        if n > 0:
            out[b, h, :n] = normal_f32(seed, tensor_id, (n, d), part=bh)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(B * H)))
    return out


def to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).to(torch.bfloat16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a CPU/GPU tensor (bf16 or fp32 values are exact in f64)."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


# ---------------------------------------------------------------------------


@dataclass
class AttnCase:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    scale: float
    causal: bool
    key_len: Optional[torch.Tensor]  # int32 [B] or None (= Nk)
    name: str = ""
    meta: dict = field(default_factory=dict)


def single_query(seed: int = 1, n: int = 4096, d: int = 64):
    q = torch.from_numpy(normal_f32(seed, _Q, (d,)))
    k = torch.from_numpy(normal_f32(seed, _K, (n, d)))
    v = torch.from_numpy(normal_f32(seed, _V, (n, d)))
    return q, k, v, 1.0


def softmax_logits(seed: int = 2, rows: int = 4096, cols: int = 32768,
                   sigma: float = 2.0, spike_frac: float = 0.01,
                   spike: float = 40.0) -> torch.Tensor:
    """fp32 [rows, cols]; entries sigma*N(0,1), round(spike_frac*rows*cols) set to spike."""
    x = np.empty((rows, cols), dtype=np.float32)
    nparts = max(1, min(64, rows))
    bounds = np.linspace(0, rows, nparts + 1).astype(np.int64)

    def work(p):
        r0, r1 = bounds[p], bounds[p + 1]
        if r1 > r0:
            x[r0:r1] = normal_f32(seed, _X, (r1 - r0, cols), part=p, sigma=sigma)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nparts)))
    nspike = int(round(spike_frac * rows * cols))
    if nspike:
        pos = _gen(seed, _SPIKE).choice(rows * cols, size=nspike, replace=False)
        x.reshape(-1)[pos] = np.float32(spike)
    return torch.from_numpy(x)


def key_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Per-batch valid key lengths, uniform integers on [lo, hi]."""
    return _gen(seed, _LEN).integers(lo, hi + 1, size=B).astype(np.int32)


def attention(seed: int, B: int, H: int, Nq: int, Nk: int, d: int, causal: bool,
              len_range=None, name: str = "") -> AttnCase:
    lens = key_lengths(seed, B, *len_range) if len_range is not None else None
    q = to_bf16(normal_bhnd(seed, _Q, B, H, Nq, d))
    k = to_bf16(normal_bhnd(seed, _K, B, H, Nk, d))
    v = to_bf16(normal_bhnd(seed, _V, B, H, Nk, d))
    kl = torch.from_numpy(lens) if lens is not None else None
    return AttnCase(q, k, v, 1.0 / math.sqrt(d), causal, kl, name=name)


def attention_dominant_keys(seed: int, B: int, H: int, N: int, d: int, causal: bool,
                            beta_range=(1.0, 4.0), v_range=(4.0, 6.0)) -> AttnCase:
    """Nearly one-hot rows whose dominant key lies in a late key tile.

    K is N(0,1).  Query row i is beta_i times one key t(i) (beta_i uniform on
    ``beta_range``): t(i) = i when causal (the diagonal key, in the row's last
    key tile), else a key of the last 128-key tile.  So s_i,t(i) ~ beta_i |k|^2
    / sqrt(d) stands about beta_i * (sqrt(d) - 3) above the other scores.  V
    entries have random signs and magnitudes uniform on ``v_range``.  Returns
    the case and t as an int64 array [N].
    """
    k = to_bf16(normal_bhnd(seed, _K, B, H, N, d))
    i = np.arange(N)
    t = i.copy() if causal else (N - 1 - (i % min(N, 128)))
    g = _gen(seed, _Q)
    beta = g.uniform(*beta_range, size=(B, H, N, 1)).astype(np.float32)
    q = to_bf16(k.float().numpy()[:, :, t, :] * beta)
    gv = _gen(seed, _V)
    mag = gv.uniform(*v_range, size=(B, H, N, d)).astype(np.float32)
    sign = np.where(gv.random(size=(B, H, N, d)) < 0.5, -1.0, 1.0).astype(np.float32)
    v = to_bf16(mag * sign)
    case = AttnCase(q, k, v, 1.0 / math.sqrt(d), causal, None,
                    name=f"dominant keys B{B} H{H} N{N} d{d} causal={causal}")
    case.meta["target"] = t
    return case


def attn(seed: int = 3) -> AttnCase:
    return attention(seed, 4, 16, 4096, 4096, 128, False, None, "attn B4 H16 N4096 d128")


def attn_causal(seed: int = 4) -> AttnCase:
    return attention(seed, 8, 32, 8192, 8192, 128, True, (4096, 8192),
                     "attn causal+padding B8 H32 N8192 d128")


@dataclass
class DecodeCase:
    q: torch.Tensor          # [B, H, 1, d]
    k: torch.Tensor          # [B, H, Nk, d]
    v: torch.Tensor
    key_len: torch.Tensor    # int32 [B]
    scale: float
    num_splits: int
    name: str = ""


def decode(seed: int = 5, B: int = 64, H: int = 32, Nk: int = 32768, d: int = 128,
           len_range=(1024, 32768), num_splits: int = 16, spike_frac: float = 0.001,
           spike_mult: float = 8.0, device: str = "cpu",
           keep_host: Sequence[int] = ()) -> DecodeCase:
    """Split-KV decode inputs, generated one batch entry at a time.

    With device="cuda" each batch entry is generated on the host, rounded to
    bf16 and copied into a device tensor, so host memory stays at one entry.
    ``keep_host``: batch indices whose host bf16 K/V are kept for the oracle in
    ``case.meta_host`` as {b: (k_b, v_b)}.
    """
    lens = key_lengths(seed, B, *len_range)
    q = to_bf16(normal_bhnd(seed, _Q, B, H, 1, d))
    nspike = int(round(spike_frac * B * H * Nk))
    spike_pos = _gen(seed, _SPIKE).choice(B * H * Nk, size=nspike, replace=False)
    sb, rem = np.divmod(spike_pos, H * Nk)
    sh, sj = np.divmod(rem, Nk)
    k = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device=device)
    v = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device=device)
    host = {}
    for b in range(B):
        n = int(lens[b])
        kb = np.zeros((H, Nk, d), dtype=np.float32)
        vb = np.zeros((H, Nk, d), dtype=np.float32)

        def work(h):
            kb[h, :n] = normal_f32(seed, _K, (n, d), part=b * H + h)
            vb[h, :n] = normal_f32(seed, _V, (n, d), part=b * H + h)

        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(H)))
        sel = sb == b
        kb[sh[sel], sj[sel]] *= np.float32(spike_mult)
        kb16, vb16 = to_bf16(kb), to_bf16(vb)
        k[b].copy_(kb16)
        v[b].copy_(vb16)
        if b in keep_host:
            host[b] = (kb16, vb16)
    case = DecodeCase(q.to(device), k, v, torch.from_numpy(lens).to(device),
                      1.0 / math.sqrt(d), num_splits,
                      name=f"decode B{B} H{H} Nk{Nk} d{d} splits{num_splits}")
    case.meta_host = host
    return case
