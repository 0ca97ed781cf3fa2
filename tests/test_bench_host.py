"""Host-side logic of bench.py: algorithmic work counts and the max-over-ranks
reduction (world size 2 over gloo on the CPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle


def test_attn_flops_counts_visible_pairs():
    # brute force over tiny shapes with the oracle's visibility rule
    for B, Nq, Nk, causal in ((2, 5, 7, True), (2, 7, 5, True), (3, 6, 6, False)):
        kl = [Nk, 2, 0][:B]
        want = 0
        for b in range(B):
            for i in range(Nq):
                want += oracle.visible_keys(i, Nq, Nk, causal, kl[b])
        assert bench.attn_flops(B, 3, Nq, Nk, 16, causal, kl) == 4 * 16 * 3 * want


def test_workload_sizes():
    assert bench.attn_flops(4, 16, 4096, 4096, 128, False, None) == 549_755_813_888
    full_causal = bench.attn_flops(8, 32, 8192, 8192, 128, True, [8192] * 8)
    assert full_causal == 4 * 128 * 32 * 8 * 8192 * 8193 // 2
    assert bench.decode_bytes(2, 3, 128, [10, 20]) == 3 * 30 * 128 * 2 * 2 + 2 * 3 * 128 * 2 * 2 + 2 * 3 * 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = {"attn_ms": 1.0 + rank, "soft_ms": 5.0 - rank, "total_ms": 2.0}
    out = bench.reduce_max(times, world, "cpu")
    q.put((rank, out))
    dist.destroy_process_group()


def test_reduce_max_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert got[r] == {"attn_ms": 2.0, "soft_ms": 5.0, "total_ms": 2.0}


def test_reduce_max_single_rank_is_identity():
    assert bench.reduce_max({"a": 1.5}, 1, "cpu") == {"a": 1.5}


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_sampler_keeps_readings_inside_the_timed_region():
    import datetime
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = []
    for i, (mhz, w, pcap) in enumerate([(1500, 150, "Not Active"), (2070, 900, "Not Active"),
                                        (2070, 1100, "Active"), (1600, 160, "Not Active")]):
        ts = (base + datetime.timedelta(milliseconds=20 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, 0, {mhz}, 2070, {w}, 0x0, Not Active, Not Active, Not Active, {pcap}")
    c = bench.ClockSampler(0)
    c.proc = _FakeProc("\n".join(lines) + "\n")
    t0 = (base + datetime.timedelta(milliseconds=10)).timestamp()
    t1 = (base + datetime.timedelta(milliseconds=50)).timestamp()
    r = c.stop(t0, t1)
    assert r["samples"] == 2 and r["samples_in_timed_region"] == 2
    assert r["sm_mhz"] == 2070 and r["power_w_max"] == 1100 and r["reasons"] == ["sw_power_cap"]
    # a region shorter than the reading interval keeps the first reading after its start
    c.proc = _FakeProc("\n".join(lines) + "\n")
    t0 = (base + datetime.timedelta(milliseconds=25)).timestamp()
    r = c.stop(t0, t0 + 0.001)
    assert r["samples"] == 1 and r["samples_in_timed_region"] == 0 and r["power_w_max"] == 1100
