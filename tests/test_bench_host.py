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
