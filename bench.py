"""Benchmark of the exact online-softmax attention hot path on one GB300.

One step = one pass of every hot-path operation over its synthetic workload:
  attention forward  B8 H32 N8192 d128 bf16, causal, key_len ~ U[4096, 8192]
  row softmax        4096 x 32768 fp32 (2*N(0,1), 1% of entries at +40)
  split-KV decode    B64 H32 Nk32768 d128 bf16, 16 splits, key_len ~ U[1024, 32768],
                     followed by the merge of the split summaries
The JSON line's headline `value` is the attention forward's throughput
(algorithmic TFLOP/s: 4*d per visible (query, key) pair, exponentials not
counted); the softmax and decode throughputs (algorithmic GB/s) are reported
under "components", each with its own roofline.  All inputs are larger than
the 129 MB L2, so no flush runs between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl osm|reference]

--impl reference times the float64 CPU oracle (the reference arm of this
method) on a bounded sample of the same attention workload.
Under torchrun each rank runs the same per-GPU work (weak scaling); rank 0
prints the line with the maximum time over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOPS & % BF16 tensor peak; softmax/decode GB/s & % HBM peak"
CSRC = os.path.join(ROOT, "exact_tiled_attention_osm_gb300", "csrc")

# DRAM traffic of one launch on the bench workload from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, summed over the kernels of the
# operation), valid only for the kernel sources it was captured on (sha256 of
# the listed files, concatenated); None until captured on the current source.
KERNEL_TRAFFIC = {
    # attn_fwd_kernel<false, 128>, causal+padding B8 H32 N8192: read 1,335,807,744
    # + write 519,688,192
    "attn_fwd_kernel": {"bytes_per_launch": 1_335_807_744 + 519_688_192,
                        "sources": ["attn_fwd.cu", "ptx.cuh"],
                        "source_sha256": "6ff9ae89e7ceca73af8091b19a4c919b3cc91c9db1e7abea1253f029c687dceb"},
    # softmax_rows_cluster<8>, 4096 x 32768: read 536,921,088 + write 482,430,208
    "softmax_rows": {"bytes_per_launch": 536_921_088 + 482_430_208,
                     "sources": ["softmax_rows.cu", "exp_le0.cuh", "ptx.cuh"],
                     "source_sha256": "c84597e1141cf857b1bb5c183ced97a033a0280f8a9e4888cdb55ade18b7b39e"},
    # decode_split_kernel read 17,360,717,824 + write 11,526,144;
    # merge_kernel read 17,050,880 + write 0
    "decode_splitkv": {"bytes_per_launch": 17_360_717_824 + 11_526_144 + 17_050_880,
                       "sources": ["decode.cu", "ptx.cuh"],
                       "source_sha256": "1fd03b86d792f286b8134d7190d3a05277e35f93f34299ed11b71fd7216c61a7"},
}


def captured_traffic(kernel):
    t = KERNEL_TRAFFIC[kernel]
    h = hashlib.sha256()
    for name in t["sources"]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return t["bytes_per_launch"] if h.hexdigest() == t["source_sha256"] else None


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- algorithmic work

def attn_flops(B, H, Nq, Nk, d, causal, key_len):
    """4*d per visible (query, key) pair: 2*d for q.k and 2*d for p*v."""
    tot = 0
    for b in range(B):
        L = min(max(int(key_len[b]) if key_len is not None else Nk, 0), Nk)
        if causal:
            off = Nk - Nq
            i = np.arange(Nq, dtype=np.int64)
            vis = np.clip(np.minimum(L, i + 1 + off), 0, None)
            tot += int(vis.sum())
        else:
            tot += L * Nq
    return 4 * d * H * tot


def decode_bytes(B, H, d, key_len, elem=2):
    keys = sum(int(x) for x in key_len)
    return H * keys * d * elem * 2 + B * H * d * elem * 2 + B * H * 4


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi readings every 20 ms; stop() keeps the ones taken inside the
    timed region (wall clock, from the first launch to the final
    synchronisation), or the nearest one after its start when the region is
    shorter than a reading."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]),
                             {nm for nm, val in zip(names, parts[6:10]) if val.lower() == "active"}))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        if not inside and t0 is not None:
            after = [r for r in rows if r[0] >= t0]
            inside = after[:1]
        use = inside if inside else rows
        reasons = set().union(*[r[4] for r in use]) if use else set()
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": use[-1][2] if use else None,
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len([r for r in rows if t0 is not None and t0 <= r[0] <= t1]),
                "power_w_max": max(r[3] for r in use) if use else None}


# ----------------------------------------------------------------- the GPU arm

class Workloads:
    def __init__(self, dev):
        import workloads as W
        t0 = time.time()
        self.attn = W.attn_causal()
        a = self.attn
        self.q, self.k, self.v = a.q.to(dev), a.k.to(dev), a.v.to(dev)
        self.kl = a.key_len.to(dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(a.q.shape[:3], dtype=torch.float32, device=dev)
        B, H, N, d = a.q.shape
        self.attn_flops = attn_flops(B, H, N, N, d, True, a.key_len.numpy())
        x = W.softmax_logits(2)
        self.x = x.to(dev)
        self.y = torch.empty_like(self.x)
        self.softmax_bytes = 8 * x.numel()
        dc = W.decode(5, device=str(dev))
        self.dec = dc
        from exact_tiled_attention_osm_gb300 import decode_workspace_bytes
        Bd, Hd, _, dd = dc.q.shape
        self.ws = torch.empty(decode_workspace_bytes(Bd, Hd, dd, dc.num_splits), dtype=torch.uint8,
                              device=dev)
        self.od = torch.empty_like(dc.q)
        self.ld = torch.empty((Bd, Hd), dtype=torch.float32, device=dev)
        self.decode_bytes = decode_bytes(Bd, Hd, dd, dc.key_len.cpu().numpy())
        self.setup_s = time.time() - t0


def gpu_arm(args, rank, world, dev):
    import exact_tiled_attention_osm_gb300 as osm
    osm.load_library()
    wl = Workloads(dev)
    stream = torch.cuda.current_stream(dev)
    dc = wl.dec

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        osm.attn_fwd(wl.q, wl.k, wl.v, wl.attn.scale, True, wl.kl, out=wl.o, lse=wl.lse)
        if ev is not None:
            ev[1].record(stream)
        osm.softmax_rows(wl.x, out=wl.y)
        if ev is not None:
            ev[2].record(stream)
        osm.attn_decode_splitkv(dc.q, dc.k, dc.v, dc.scale, dc.key_len, dc.num_splits,
                                workspace=wl.ws, out=wl.od, lse=wl.ld)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if osm.device_status() != 0:
        raise RuntimeError("a device-side wait ran out during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clk = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clk.start()
    time.sleep(0.3)  # let the sampler take its first reading
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop(t_wall0, t_wall1)
    total_ms = start.elapsed_time(end)
    t_attn = [e[0].elapsed_time(e[1]) for e in evs]
    t_soft = [e[1].elapsed_time(e[2]) for e in evs]
    t_dec = [e[2].elapsed_time(e[3]) for e in evs]
    if osm.device_status() != 0:
        raise RuntimeError("a device-side wait ran out during the timed region")

    # End to end through the public API with host buffers.  Every step copies
    # its attention inputs from pinned host memory (H2D), calls attn_fwd and
    # reads O and LSE back (D2H).  Steps are pipelined the way a caller would
    # stream batches: two device buffer sets, the copies on their own streams,
    # so step s+1's H2D and step s-1's D2H overlap step s's kernel (the link
    # carries both directions at once).  Events order every buffer reuse.
    hq, hk, hv = (t.pin_memory() for t in (wl.attn.q, wl.attn.k, wl.attn.v))
    hkl = wl.attn.key_len.pin_memory()
    ho = [torch.empty(wl.o.shape, dtype=wl.o.dtype, pin_memory=True) for _ in range(2)]
    hl = [torch.empty(wl.lse.shape, dtype=wl.lse.dtype, pin_memory=True) for _ in range(2)]
    dbuf = [(wl.q, wl.k, wl.v, wl.kl),
            (torch.empty_like(wl.q), torch.empty_like(wl.k), torch.empty_like(wl.v),
             torch.empty_like(wl.kl))]
    obuf = [(wl.o, wl.lse), (torch.empty_like(wl.o), torch.empty_like(wl.lse))]
    ev = lambda: torch.cuda.Event()
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_free = [ev(), ev()]    # the kernel that read input set b has finished
    in_ready = [ev(), ev()]   # input set b copied
    out_ready = [ev(), ev()]  # output set b written
    out_free = [ev(), ev()]   # output set b copied back
    for b in range(2):
        in_free[b].record(stream)
        out_free[b].record(stream)

    def e2e_step(i):
        b = i & 1
        dq, dk, dv, dkl = dbuf[b]
        o, lse = obuf[b]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(in_free[b])
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dkl.copy_(hkl, non_blocking=True)
            in_ready[b].record(s_h2d)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        osm.attn_fwd(dq, dk, dv, wl.attn.scale, True, dkl, out=o, lse=lse)
        in_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(out_ready[b])
            ho[b].copy_(o, non_blocking=True)
            hl[b].copy_(lse, non_blocking=True)
            out_free[b].record(s_d2h)

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)  # before the first timed H2D: the copy stream waits on it
    s_h2d.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(out_free[(e2e_steps - 1) & 1])  # the last D2H has landed
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hkl))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    del hq, hk, hv, ho, hl, dbuf, obuf

    res = {
        "total_ms": total_ms,
        "attn_ms": statistics.mean(t_attn),
        "soft_ms": statistics.mean(t_soft),
        "dec_ms": statistics.mean(t_dec),
        "e2e_ms": e2e_ms,
        "h2d": h2d, "d2h": d2h,
        "clocks": clocks,
        "setup_s": wl.setup_s,
        "attn_flops": wl.attn_flops,
        "softmax_bytes": wl.softmax_bytes,
        "decode_bytes": wl.decode_bytes,
    }
    return res


def cpu_oracle_sample(budget_s=12.0, seed_rows=0):
    """Time the float64 oracle on (b, h) heads of the attention workload, 1024
    query rows each, until `budget_s` of CPU time is spent.  Returns
    (TFLOP/s, description, threads)."""
    import oracle
    import workloads as W
    B, H, N, d = 8, 32, 8192, 128
    lens = W.key_lengths(4, B, 4096, 8192)
    rng = np.random.default_rng(seed_rows)
    flops, t_used, heads = 0, 0.0, 0
    # generate one head at a time (the oracle's inputs are the same bf16 values)
    for idx in range(B * H):
        b, h = divmod((idx * 37) % (B * H), H)
        part = b * H + h
        q = W.to_bf16(W.normal_f32(4, 1, (N, d), part=part))
        k = W.to_bf16(W.normal_f32(4, 2, (N, d), part=part))
        v = W.to_bf16(W.normal_f32(4, 3, (N, d), part=part))
        rows = np.sort(rng.choice(N, size=1024, replace=False))
        q64, k64, v64 = (W.as_f64(t)[None, None] for t in (q, k, v))
        t0 = time.perf_counter()
        oracle.attention_ref(q64, k64, v64, 1 / math.sqrt(d), True, [int(lens[b])], rows=rows)
        t_used += time.perf_counter() - t0
        L = int(lens[b])
        flops += 4 * d * int(np.minimum(L, rows + 1).sum())
        heads += 1
        if t_used >= budget_s:
            break
    desc = (f"{heads} (b,h) heads x 1024 sampled query rows of the causal+padding "
            f"B8 H32 N8192 d128 workload, all their visible keys")
    return flops / t_used / 1e12, desc, t_used


def oracle_step(idx, rows_per_step=256):
    """One step of the reference arm: the float64 oracle on one (b, h) head of
    the causal+padding workload (heads taken in a fixed scattered order),
    `rows_per_step` sampled query rows with all their visible keys.  Input
    generation is outside the timed part.  Returns (FLOPs, seconds)."""
    import oracle
    import workloads as W
    B, H, N, d = 8, 32, 8192, 128
    lens = W.key_lengths(4, B, 4096, 8192)
    b, h = divmod((idx * 37) % (B * H), H)
    part = b * H + h
    q = W.to_bf16(W.normal_f32(4, 1, (N, d), part=part))
    k = W.to_bf16(W.normal_f32(4, 2, (N, d), part=part))
    v = W.to_bf16(W.normal_f32(4, 3, (N, d), part=part))
    rows = np.sort(np.random.default_rng(idx).choice(N, size=rows_per_step, replace=False))
    q64, k64, v64 = (W.as_f64(t)[None, None] for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.attention_ref(q64, k64, v64, 1 / math.sqrt(d), True, [int(lens[b])], rows=rows)
    dt = time.perf_counter() - t0
    return 4 * d * int(np.minimum(int(lens[b]), rows + 1).sum()), dt


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


TIME_KEYS = ("total_ms", "attn_ms", "soft_ms", "dec_ms", "e2e_ms")


def reduce_max(times: dict, world: int, device) -> dict:
    """Element-wise maximum of a dict of times over all ranks (identity at world 1)."""
    keys = sorted(times)
    t = torch.tensor([float(times[k]) for k in keys], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return dict(zip(keys, t.tolist()))


def profile_case(spec: str, iters: int):
    """Run one operation `iters` times on a given shape (for ncu captures).

    spec: "attn:B,H,N[,causal][,d64]" | "attnnorm:B,H,N[,causal][,d64]" (the normalised
          form) | "attnqk:B,H,N[,causal]" (QK-norm inputs with
          their score bound) | "bwd:B,H,N[,causal][,d64]" | "softmax:rows,cols"
          | "topk:rows,cols,k[,nospike]"
          | "decode:B,H,Nk[,splits]"
          | "append:B,H,Nk,n_new[,splits]" | "lsemerge:S,rows,d".
    Inputs come from the same generators as the full workloads.
    """
    import exact_tiled_attention_osm_gb300 as osm
    import workloads as W
    op, _, arg = spec.partition(":")
    parts = arg.split(",")
    dev = torch.device("cuda", 0)
    if op in ("attn", "attnnorm"):
        # attnnorm: the normalised form (one division per key tile)
        B, H, N = (int(x) for x in parts[:3])
        causal = "causal" in parts[3:]
        hd = 64 if "d64" in parts[3:] else 128
        c = W.attention(4, B, H, N, N, hd, causal, (N // 2, N) if causal else None)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        kl = c.key_len.to(dev) if c.key_len is not None else None
        norm = op == "attnnorm"
        run = lambda: osm.attn_fwd(q, k, v, c.scale, causal, kl, normalised=norm)
        work = attn_flops(B, H, N, N, hd, causal, None if kl is None else c.key_len.numpy())
        unit = "TFLOP/s"
    elif op == "attnqk":
        # QK-norm inputs (q, k rows scaled to norm sqrt(d)) with their known
        # score bound scale * max|q| * max|k|, through osm_attn_fwd_bounded
        B, H, N = (int(x) for x in parts[:3])
        causal = len(parts) > 3 and parts[3] == "causal"
        c = W.attention(4, B, H, N, N, 128, causal, (N // 2, N) if causal else None)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        q = (q.float() / q.float().norm(dim=-1, keepdim=True) * 128 ** 0.5).to(torch.bfloat16)
        k = (k.float() / k.float().norm(dim=-1, keepdim=True) * 128 ** 0.5).to(torch.bfloat16)
        bound = c.scale * float(q.float().norm(dim=-1).max()) * float(k.float().norm(dim=-1).max())
        kl = c.key_len.to(dev) if c.key_len is not None else None
        run = lambda: osm.attn_fwd(q, k, v, c.scale, causal, kl, score_bound=bound)
        work = attn_flops(B, H, N, N, 128, causal, None if kl is None else c.key_len.numpy())
        unit = "TFLOP/s"
    elif op == "bwd":
        # attention backward; O and lse from the forward kernel on the same inputs
        B, H, N = (int(x) for x in parts[:3])
        causal = "causal" in parts[3:]
        hd = 64 if "d64" in parts[3:] else 128
        c = W.attention(4, B, H, N, N, hd, causal, (N // 2, N) if causal else None)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        kl = c.key_len.to(dev) if c.key_len is not None else None
        o, lse = osm.attn_fwd(q, k, v, c.scale, causal, kl)
        do = W.to_bf16(W.normal_bhnd(4, 7, B, H, N, hd)).to(dev)
        ws = torch.empty(osm.attn_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device=dev)
        run = lambda: osm.attn_bwd(q, k, v, o, lse, do, c.scale, causal, kl, workspace=ws)
        # 5 products of 2 d FLOPs per visible (query, key) pair = 2.5 x the forward's
        work = 2.5 * attn_flops(B, H, N, N, hd, causal,
                                None if kl is None else c.key_len.numpy())
        unit = "TFLOP/s"
    elif op == "softmax":
        R, C = (int(x) for x in parts[:2])
        x = W.softmax_logits(2, rows=R, cols=C).to(dev)
        y = torch.empty_like(x)
        run = lambda: osm.softmax_rows(x, out=y)
        work, unit = 8 * R * C, "GB/s"
    elif op == "topk":
        R, C, kk = (int(x) for x in parts[:3])
        spikes = 0.0 if "nospike" in parts[3:] else 0.01  # the workload's 1 % of entries at 40.0
        x = W.softmax_logits(2, rows=R, cols=C, spike_frac=spikes).to(dev)
        ii = torch.empty((R, kk), dtype=torch.int32, device=dev)
        pp = torch.empty((R, kk), dtype=torch.float32, device=dev)
        run = lambda: osm.softmax_topk(x, kk, idx=ii, prob=pp)
        work, unit = 4 * R * C + 8 * R * kk, "GB/s"
    elif op == "decode":
        B, H, Nk = (int(x) for x in parts[:3])
        S = int(parts[3]) if len(parts) > 3 else 16
        dc = W.decode(5, B=B, H=H, Nk=Nk, len_range=(Nk // 32, Nk), num_splits=S, device="cuda")
        ws = torch.empty(osm.decode_workspace_bytes(B, H, 128, S), dtype=torch.uint8, device=dev)
        run = lambda: osm.attn_decode_splitkv(dc.q, dc.k, dc.v, dc.scale, dc.key_len, S,
                                              workspace=ws)
        work, unit = decode_bytes(B, H, 128, dc.key_len.cpu().numpy()), "GB/s"
    elif op == "append":
        # extend running summaries by the last n_new keys of a B x H x Nk cache
        B, H, Nk, n_new = (int(x) for x in parts[:4])
        S = int(parts[4]) if len(parts) > 4 else 16
        dc = W.decode(5, B=B, H=H, Nk=Nk, len_range=(Nk, Nk), num_splits=S, device="cuda")
        ws = torch.empty(osm.decode_append_workspace_bytes(B, H, 128, S), dtype=torch.uint8,
                         device=dev)
        state = osm.decode_state(B, H, 128, dev)
        ks = torch.full((B,), Nk - n_new, dtype=torch.int32, device=dev)
        osm.attn_decode_append(dc.q, dc.k, dc.v, state, None, ks, dc.scale, S, workspace=ws)
        run = lambda: osm.attn_decode_append(dc.q, dc.k, dc.v, state, ks, None, dc.scale, S,
                                             workspace=ws)
        # new K/V rows + q + o (bf16) + lse + the state read and written (fp32)
        work = (B * H * n_new * 128 * 2 * 2 + B * H * 128 * 2 * 2 + B * H * 4
                + 2 * B * H * (128 + 2) * 4)
        unit = "GB/s"
    elif op == "lsemerge":
        # LSE-form merge of S normalised partials of rows x d (fp32 in, bf16 out)
        S, R, d = (int(x) for x in parts[:3])
        g = torch.Generator(device="cpu").manual_seed(6)
        op_ = torch.randn((S, R, d), generator=g).to(dev)
        lp = (torch.randn((S, R), generator=g) * 3).to(dev)
        run = lambda: osm.lse_merge(op_, lp, torch.bfloat16)
        work, unit = S * R * (d + 1) * 4 + R * (d * 2 + 4), "GB/s"
    else:
        raise SystemExit(f"unknown op {op}")
    run()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * iters)]
    for i in range(iters):
        ev[2 * i].record()
        run()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    if osm.device_status() != 0:
        raise RuntimeError("a device-side wait ran out")
    ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(iters)]
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"profile": spec, "iters": iters, "ms": ms,
                      "best": work / (min(ms) * 1e-3) / scale, "unit": unit, "work": work}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="osm", choices=["osm", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="run one op on a given shape instead of the benchmark, e.g. "
                         "attn:2,16,8192,causal | softmax:1024,32768 | decode:4,32,32768")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        profile_case(args.profile, args.iters)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pk, pk_kind = peaks()
    config = {"workload": "attn fwd causal+padding B8 H32 N8192 d128 bf16 (key_len U[4096,8192]); "
                          "softmax 4096x32768 fp32; decode B64 H32 Nk32768 d128 bf16 16 splits",
              "attn": {"B": 8, "H": 32, "Nq": 8192, "Nk": 8192, "d": 128, "causal": True,
                       "key_len": "U[4096,8192]", "scale": "1/sqrt(128)"},
              "softmax": {"rows": 4096, "cols": 32768},
              "decode": {"B": 64, "H": 32, "Nk": 32768, "d": 128, "num_splits": 16,
                         "key_len": "U[1024,32768]"},
              "l2": "inputs larger than L2 (129 MB); no flush between steps",
              "parallelism": f"replicas x{args.gpus}"}

    if args.impl == "reference":
        if rank != 0:
            return
        # W untimed warm-up steps, then K timed steps, each a bounded sample
        for i in range(args.warmup):
            oracle_step(10_000 + i)
        flops, secs = 0, 0.0
        for i in range(args.steps):
            f, dt = oracle_step(i)
            flops += f
            secs += dt
        tf = flops / secs / 1e12
        desc = (f"{args.steps} steps, each one (b,h) head x 256 sampled query rows of the "
                f"causal+padding B8 H32 N8192 d128 workload with all their visible keys")
        cores = blas_threads()
        line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
                "config": config,
                "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": cores,
                                 "kind": "oracle", "sample": desc},
                "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libosm has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    res = gpu_arm(args, rank, world, dev)

    # max over ranks of every time; per-GPU work is identical (weak scaling)
    mx = reduce_max({k: res[k] for k in TIME_KEYS}, world, dev)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    attn_tf = world * res["attn_flops"] / (mx["attn_ms"] * 1e-3) / 1e12
    soft_gbs = world * res["softmax_bytes"] / (mx["soft_ms"] * 1e-3) / 1e9
    dec_gbs = world * res["decode_bytes"] / (mx["dec_ms"] * 1e-3) / 1e9
    per_gpu_tf = attn_tf / world
    traffic = captured_traffic("attn_fwd_kernel")
    peak_tc = pk["bf16_tflops"]
    roofline = {"bound": "tensor", "achieved": per_gpu_tf, "peak": peak_tc, "unit": "TFLOP/s",
                "frac": per_gpu_tf / peak_tc, "traffic": traffic,
                "peak_kind": f"{pk_kind} bf16 burst",
                "frac_of_sustained": per_gpu_tf / pk.get("bf16_tflops_sustained", peak_tc),
                "kernel": "attn_fwd_kernel", "per_launch_flops": res["attn_flops"],
                "avg_launch_ms": mx["attn_ms"]}
    hbm = pk["hbm_gbs"]
    components = {
        "softmax_rows": {"value": soft_gbs, "unit": "GB/s", "ms": mx["soft_ms"],
                         "roofline": {"bound": "hbm", "achieved": soft_gbs / world, "peak": hbm,
                                      "unit": "GB/s", "frac": soft_gbs / world / hbm,
                                      "traffic": captured_traffic("softmax_rows"),
                                      "per_launch_bytes": res["softmax_bytes"],
                                      "peak_kind": f"{pk_kind} copy"}},
        "decode_splitkv": {"value": dec_gbs, "unit": "GB/s", "ms": mx["dec_ms"],
                           "roofline": {"bound": "hbm", "achieved": dec_gbs / world, "peak": hbm,
                                        "unit": "GB/s", "frac": dec_gbs / world / hbm,
                                        "traffic": captured_traffic("decode_splitkv"),
                                        "per_launch_bytes": res["decode_bytes"],
                                        "peak_kind": f"{pk_kind} copy",
                                        "note": "split kernel + merge kernel, one pass"}},
    }
    e2e_tf = world * res["attn_flops"] / (mx["e2e_ms"] * 1e-3) / 1e12
    line = {"metric": METRIC, "value": attn_tf, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mx["total_ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, generated on the host)", "config": config,
            "roofline": roofline, "components": components,
            "e2e": {"value": e2e_tf, "unit": "TFLOP/s", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"], "ms_per_step": mx["e2e_ms"],
                    "what": "attention forward via the public API from pinned host buffers; each step's H2D of its inputs and D2H of O and LSE, pipelined across steps on copy streams"},
            "gpu_launches": 4 * args.steps,
            "clocks": res["clocks"]}
    if not args.no_cpu_baseline and world == 1:
        tf, desc, used = cpu_oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": blas_threads(),
                                "kind": "oracle", "sample": desc, "seconds": used}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
