"""The allocation-free decode entry point, called through the C ABI.

osm_attn_decode_splitkv_noalloc serves callers that cannot allocate device
memory (for example a plug-in whose host program owns all device memory): it
keeps the split summaries in a fixed scratch area inside libosm instead of a
caller workspace.  This file is collected last so a run that stops at the
first failure has already run every other test; it also passes on its own in
a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm
import oracle
import workloads as W
from bars import o_bar

pytestmark = pytest.mark.gpu


def _noalloc(lib, dt, q, k, v, o, lse, key_len, splits, scale):
    B, H, _, d = q.shape
    return lib.osm_attn_decode_splitkv_noalloc(
        dt, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
        k.shape[2], d, ctypes.c_float(scale), key_len.data_ptr(), splits,
        torch.cuda.current_stream().cuda_stream)


def _with_workspace(lib, dt, q, k, v, o, lse, key_len, splits, scale):
    B, H, _, d = q.shape
    need = lib.osm_attn_decode_splitkv_workspace_bytes(B, H, d, splits)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    return lib.osm_attn_decode_splitkv(
        dt, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
        k.shape[2], d, ctypes.c_float(scale), key_len.data_ptr(), splits, ws.data_ptr(), need,
        torch.cuda.current_stream().cuda_stream), ws


def _close(o, lse, o_ref, lse_ref, bf16):
    o, lse, o_ref, lse_ref = (W.as_f64(t) for t in (o, lse, o_ref, lse_ref))
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    if bf16:
        assert np.all(np.abs(o - o_ref) <= o_bar(o_ref))
        assert float(np.max(np.abs(lse[fin] - lse_ref[fin]), initial=0.0)) <= 1e-3
    else:
        assert float(np.max(np.abs(o - o_ref))) <= 1e-5
        assert float(np.max(np.abs(lse[fin] - lse_ref[fin]), initial=0.0)) <= 1e-5


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(cuda_ok):
    lib = osm.load_library()
    cases = [
        # bf16, d=128, 16 splits, one batch entry with no keys at all
        (W.decode(seed=71, B=4, H=8, Nk=3000, d=128, len_range=(1, 3000), num_splits=16),
         torch.bfloat16, osm.OSM_BF16, [0, None, None, None]),
        # fp32, d=64, a different shape and split count right after it
        (W.decode(seed=72, B=3, H=5, Nk=1500, d=64, len_range=(200, 1500), num_splits=7),
         torch.float32, osm.OSM_F32, [None, None, None]),
    ]
    for case, tdt, dt, overrides in cases:
        q, k, v = (t.to(tdt).cuda() for t in (case.q, case.k, case.v))
        kl = case.key_len.clone()
        for i, val in enumerate(overrides):
            if val is not None:
                kl[i] = val
        kl = kl.cuda()
        B, H = q.shape[:2]
        o_a = torch.empty_like(q)
        l_a = torch.empty((B, H), dtype=torch.float32, device="cuda")
        o_b, l_b = torch.empty_like(o_a), torch.empty_like(l_a)
        assert _noalloc(lib, dt, q, k, v, o_a, l_a, kl, case.num_splits, case.scale) == osm.OSM_OK
        st, _ = _with_workspace(lib, dt, q, k, v, o_b, l_b, kl, case.num_splits, case.scale)
        assert st == osm.OSM_OK
        torch.cuda.synchronize()
        _close(o_a, l_a, o_b, l_b, tdt == torch.bfloat16)
        # and both against the float64 oracle
        ro, rl = oracle.attention_ref(W.as_f64(q.cpu()), W.as_f64(k.cpu()), W.as_f64(v.cpu()),
                                      case.scale, False, kl.cpu().numpy())
        _close(o_a, l_a, torch.from_numpy(ro[:, :, 0]).reshape(o_a.shape),
               torch.from_numpy(rl[:, :, 0]), tdt == torch.bfloat16)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_ok):
    lib = osm.load_library()
    B, H, d, S = 64, 64, 128, 256   # summaries far larger than the scratch area
    need = lib.osm_attn_decode_splitkv_workspace_bytes(B, H, d, S)
    assert need > osm.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, H, 1, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, 16, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    kl = torch.full((B,), 16, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, osm.OSM_BF16, q, k, k, o, lse, kl, S, 0.1) == osm.OSM_ERR_INVALID_VALUE
