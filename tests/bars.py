"""The parity bars shared by the GPU tests, and a log of the worst errors seen.

BF16 attention (forward and decode), against the float64 oracle on the same
bf16-rounded inputs:
  O, plain bar:  |O_gpu - O_ref| <= 1e-2 on every element -- the bar exactly
       as stated for the workloads, asserted on their full-size outputs.
  O, storage bar: |O_gpu - O_ref| <= 1e-2 + 2^-8 |O_ref|, i.e. 1e-2 on the
       value before the output's own bf16 storage rounding (at most 2^-8 |O|,
       half a bf16 ulp).  Asserted on the other cases: edge shapes, rows with a
       handful of keys, sharp and growing rows.  There |O| reaches 4 to 6,
       where half an ulp alone is 0.0156, and a row concentrated on a few keys
       carries the bf16 rounding of their weights (2^-8 relative each), which
       moves O by up to 2^-8 |v_i - v_j| on top of it.
  LSE: |lse_gpu - lse_ref| <= 1e-3, and -inf exactly where the oracle has -inf.
FP32 row softmax: relative error <= 1e-5.

``record`` prints the worst errors of a named case and, when the environment
names a file in OSM_PARITY_LOG, appends them there as one JSON line.
"""
import json
import os

import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3
U_BF16 = 2.0 ** -8


def o_bar(ro, plain=False):
    """Per-element O bar: the plain bar (1e-2) or the storage bar."""
    a = np.abs(ro)
    return np.full(a.shape, O_TOL) if plain else O_TOL + U_BF16 * a


def check_attention(o, lse, ro, rl, plain=False):
    """Assert the BF16 attention bars; return (max |O err|, max |LSE err|)."""
    o, lse = np.asarray(o, np.float64), np.asarray(lse, np.float64)
    assert o.shape == ro.shape and lse.shape == rl.shape
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl)), "masked-row pattern differs"
    assert np.all(np.isfinite(o))
    err_o = np.abs(o - ro)
    excess = err_o - o_bar(ro, plain)
    worst = np.unravel_index(int(np.argmax(excess)), excess.shape) if excess.size else None
    assert excess.size == 0 or float(excess.max()) <= 0.0, (
        f"O error {float(err_o[worst]):.4g} at {worst} (|O_ref| = {abs(float(ro[worst])):.4g})")
    fin = np.isfinite(rl)
    err_l = float(np.max(np.abs(lse[fin] - rl[fin]))) if fin.any() else 0.0
    assert err_l <= LSE_TOL, f"LSE error {err_l:.4g}"
    return (float(err_o.max()) if err_o.size else 0.0), err_l


def record(name, **values):
    line = {"case": name, **{k: float(v) for k, v in values.items()}}
    print("parity", json.dumps(line))
    path = os.environ.get("OSM_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")
