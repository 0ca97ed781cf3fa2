"""Failure reporting of the bounded device waits, on the GPU, without a fault.

A wait that nothing completes must give up after its limit, leave its site
code in the error word that osm_device_status reads (OSM_ERR_TIMEOUT), and
leave the context usable: the next attention call runs and matches the
oracle.
"""
import time

import numpy as np
import pytest

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import check_attention

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported(cuda_ok):
    assert osm.device_status() == 0          # clean start
    t0 = time.perf_counter()
    osm.selftest_bounded_wait()
    word = osm.device_status()              # synchronises, then reads and clears
    elapsed = time.perf_counter() - t0
    assert word == 0x7F0000A1
    assert 0.5 < elapsed < 30.0             # the wait's limit is about a second
    assert osm.device_status() == 0          # read-and-clear
    # the context still works: a small attention call against the oracle
    c = W.attention(90, 1, 2, 300, 300, 128, True, (100, 300))
    o, lse = osm.attn_fwd(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.scale, True, c.key_len.cuda())
    assert osm.device_status() == 0
    ro, rl = oracle.attention_ref(W.as_f64(c.q), W.as_f64(c.k), W.as_f64(c.v), c.scale, True,
                                  c.key_len.numpy())
    check_attention(W.as_f64(o), W.as_f64(lse), ro, rl)
