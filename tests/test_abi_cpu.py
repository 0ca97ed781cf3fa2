"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/osm.h declares, and refuses bad arguments on the host before any
launch (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_tiled_attention_osm_gb300 as osm
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "osm.h")


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_osm_gb300 import build
    build.build()
    return osm.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(osm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("osm_softmax_rows", "osm_attn_fwd", "osm_attn_decode_splitkv",
              "osm_attn_decode_splitkv_workspace_bytes", "osm_lse_merge", "osm_status_string",
              "osm_device_status", "osm_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", osm.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (osm_[a-z0-9_]+)\b", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    # the binding's signature table covers exactly the declared functions
    assert set(osm.SIGNATURES) == set(declared_functions())


def test_status_strings_and_version(lib):
    for st in range(7):
        s = osm.status_string(st)
        assert s.startswith("OSM_")
    assert "unknown" in osm.status_string(99)
    assert lib.osm_abi_version() == 103


def test_workspace_bytes_formula(lib):
    B, H, d, S = 64, 32, 128, 16
    n = B * H * S
    a = ((n * 4 + 255) // 256) * 256
    assert osm.decode_workspace_bytes(B, H, d, S) == 2 * a + n * d * 4
    assert osm.decode_workspace_bytes(B, H, 96, S) == 0
    assert osm.decode_workspace_bytes(B, H, d, 0) == 0
    assert osm.decode_workspace_bytes(B, H, d, 257) == 0


FAKE = 0x10000  # a 16-byte aligned non-null value; never dereferenced (validation fails first)


def test_softmax_validation(lib):
    f = lib.osm_softmax_rows
    assert f(None, FAKE, 4, 4, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE, None, 4, 4, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE, FAKE, -1, 4, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE + 2, FAKE, 4, 4, None) == osm.OSM_ERR_INVALID_VALUE        # misaligned
    assert f(FAKE, FAKE + 8, 4, 4, None) == osm.OSM_ERR_INVALID_VALUE        # partial overlap
    assert f(None, None, 0, 4, None) == osm.OSM_OK                            # empty: no-op
    assert f(None, None, 4, 0, None) == osm.OSM_OK


def test_softmax_topk_validation(lib):
    f = lib.osm_softmax_topk
    assert f(None, 4, 100, 8, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE, 4, 100, 8, None, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE, 4, 100, 0, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE    # k < 1
    assert f(FAKE, 4, 5, 6, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE      # k > cols
    assert f(FAKE, 4, 100, 33, FAKE, FAKE, None) == osm.OSM_ERR_UNSUPPORTED     # k > 32
    assert f(FAKE + 2, 4, 100, 8, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(FAKE, -1, 100, 8, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert f(None, 0, 100, 8, None, None, None) == osm.OSM_OK                   # empty: no-op


@pytest.mark.parametrize("entry", ["osm_attn_fwd", "osm_attn_fwd_normalised"])
def test_attn_validation(lib, entry):
    f = getattr(lib, entry)
    ok_args = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 128, 0.088, 0, None, None]

    def call(**kw):
        a = list(ok_args)
        names = ["q", "k", "v", "o", "lse", "B", "H", "Nq", "Nk", "d", "scale", "causal", "kl", "s"]
        for key, val in kw.items():
            a[names.index(key)] = val
        return f(*a)

    assert call(q=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(k=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(o=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(lse=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(q=FAKE + 8) == osm.OSM_ERR_INVALID_VALUE
    assert call(B=-1) == osm.OSM_ERR_INVALID_VALUE
    assert call(d=96) == osm.OSM_ERR_UNSUPPORTED
    assert call(d=0) == osm.OSM_ERR_INVALID_VALUE
    assert call(Nq=(1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED   # longer than 2^30
    assert call(Nk=(1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED
    assert call(scale=0.0) == osm.OSM_ERR_INVALID_VALUE
    assert call(scale=-1.0) == osm.OSM_ERR_INVALID_VALUE
    assert call(scale=float("inf")) == osm.OSM_ERR_INVALID_VALUE
    assert call(scale=float("nan")) == osm.OSM_ERR_INVALID_VALUE
    assert call(causal=2) == osm.OSM_ERR_INVALID_VALUE
    assert call(kl=FAKE + 1) == osm.OSM_ERR_INVALID_VALUE
    assert call(B=0, q=None, k=None, v=None, o=None, lse=None) == osm.OSM_OK    # empty: no-op
    assert call(Nq=0) == osm.OSM_OK


def test_bounded_attn_validation(lib):
    f = lib.osm_attn_fwd_bounded
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 128, 0.088, 0, None, 3.0, None]

    def call(i, val):
        a = list(base)
        a[i] = val
        return f(*a)

    assert call(13, float("nan")) == osm.OSM_ERR_INVALID_VALUE     # the bound must be finite
    assert call(13, float("inf")) == osm.OSM_ERR_INVALID_VALUE
    assert call(13, 1e31) == osm.OSM_ERR_INVALID_VALUE
    assert call(0, None) == osm.OSM_ERR_INVALID_VALUE              # then the usual checks
    assert call(9, 96) == osm.OSM_ERR_UNSUPPORTED
    assert call(5, 0) == osm.OSM_OK                                 # empty: no-op


def test_bwd_validation(lib):
    f = lib.osm_attn_bwd
    need = lib.osm_attn_bwd_workspace_bytes(1, 1, 128)
    assert need == 512
    names = ["q", "k", "v", "o", "lse", "do", "dq", "dk", "dv", "B", "H", "Nq", "Nk", "d",
             "scale", "causal", "kl", "ws", "wsb", "s"]
    base = [FAKE] * 9 + [1, 1, 128, 128, 128, 0.088, 0, None, FAKE, need, None]

    def call(**kw):
        a = list(base)
        for key, val in kw.items():
            a[names.index(key)] = val
        return f(*a)

    assert call(q=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(do=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(dk=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(lse=FAKE + 2) == osm.OSM_ERR_INVALID_VALUE
    assert call(dq=FAKE + 8) == osm.OSM_ERR_INVALID_VALUE
    assert call(d=96) == osm.OSM_ERR_UNSUPPORTED
    assert call(Nq=(1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED
    assert call(Nk=(1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED
    assert call(scale=0.0) == osm.OSM_ERR_INVALID_VALUE
    assert call(causal=3) == osm.OSM_ERR_INVALID_VALUE
    assert call(ws=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(ws=FAKE + 16) == osm.OSM_ERR_INVALID_VALUE
    assert call(wsb=need - 1) == osm.OSM_ERR_INVALID_VALUE
    assert call(B=0) == osm.OSM_OK                                  # empty: no-op


def test_decode_and_merge_validation(lib):
    f = lib.osm_attn_decode_splitkv
    need = osm.decode_workspace_bytes(2, 2, 128, 4)
    base = [osm.OSM_BF16, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 1000, 128, 0.088, None, 4,
            FAKE, need, None]

    def call(i, val):
        a = list(base)
        a[i] = val
        return f(*a)

    assert call(0, 7) == osm.OSM_ERR_INVALID_VALUE           # dtype
    assert call(1, None) == osm.OSM_ERR_INVALID_VALUE        # q
    assert call(9, 96) == osm.OSM_ERR_UNSUPPORTED            # d
    assert call(8, (1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED  # Nk longer than 2^30
    assert call(12, 0) == osm.OSM_ERR_INVALID_VALUE          # num_splits
    assert call(12, 300) == osm.OSM_ERR_INVALID_VALUE
    assert call(13, None) == osm.OSM_ERR_INVALID_VALUE       # workspace
    assert call(13, FAKE + 16) == osm.OSM_ERR_INVALID_VALUE  # workspace not 256-aligned
    assert call(14, need - 1) == osm.OSM_ERR_INVALID_VALUE   # workspace too small
    assert call(10, 0.0) == osm.OSM_ERR_INVALID_VALUE        # scale
    m = lib.osm_lse_merge
    assert m(None, FAKE, 2, 4, 128, osm.OSM_F32, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert m(FAKE, FAKE, 0, 4, 128, osm.OSM_F32, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert m(FAKE, FAKE, 2, 4, 100, osm.OSM_F32, FAKE, FAKE, None) == osm.OSM_ERR_UNSUPPORTED
    assert m(FAKE, FAKE, 2, 4, 128, 5, FAKE, FAKE, None) == osm.OSM_ERR_INVALID_VALUE
    assert m(FAKE, FAKE, 2, 0, 128, osm.OSM_F32, FAKE, FAKE, None) == osm.OSM_OK


def test_append_validation(lib):
    f = lib.osm_attn_decode_append
    need = osm.decode_append_workspace_bytes(2, 2, 128, 4)
    # partial summaries as for split decode, then one ticket per (b, h) row
    assert need == osm.decode_workspace_bytes(2, 2, 128, 4) + 256
    assert osm.decode_append_workspace_bytes(2, 2, 96, 4) == 0
    names = ["dt", "q", "k", "v", "B", "H", "Nk", "d", "scale", "ks", "ke", "m", "l", "o~",
             "o", "lse", "S", "ws", "wsb", "s"]
    base = [osm.OSM_BF16, FAKE, FAKE, FAKE, 2, 2, 1000, 128, 0.088, None, None, FAKE, FAKE, FAKE,
            FAKE, FAKE, 4, FAKE, need, None]

    def call(**kw):
        a = list(base)
        for key, val in kw.items():
            a[names.index(key)] = val
        return f(*a)

    assert call(dt=7) == osm.OSM_ERR_INVALID_VALUE
    assert call(q=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(m=None) == osm.OSM_ERR_INVALID_VALUE       # the state is required
    assert call(l=None) == osm.OSM_ERR_INVALID_VALUE
    assert call(**{"o~": None}) == osm.OSM_ERR_INVALID_VALUE
    assert call(m=FAKE + 2) == osm.OSM_ERR_INVALID_VALUE   # misaligned state
    assert call(ks=FAKE + 1) == osm.OSM_ERR_INVALID_VALUE
    assert call(d=96) == osm.OSM_ERR_UNSUPPORTED
    assert call(Nk=(1 << 30) + 1) == osm.OSM_ERR_UNSUPPORTED
    assert call(S=0) == osm.OSM_ERR_INVALID_VALUE
    assert call(ws=FAKE + 16) == osm.OSM_ERR_INVALID_VALUE
    assert call(wsb=need - 1) == osm.OSM_ERR_INVALID_VALUE
    assert call(scale=float("nan")) == osm.OSM_ERR_INVALID_VALUE
    assert call(B=0, q=None, m=None, l=None, ws=None) == osm.OSM_OK   # empty: no-op


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        osm.softmax_rows(torch.zeros(2, 4))
    q = torch.zeros(1, 1, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        osm.attn_fwd(q, q, q)


def test_device_status_rejects_null(lib):
    assert lib.osm_device_status(None, None) == osm.OSM_ERR_INVALID_VALUE


def test_checked_build_exports_the_same_symbols():
    """The OSM_CHECKED build compiles (here, without a GPU) and exports every
    function the header declares."""
    from exact_tiled_attention_osm_gb300 import build
    path = build.build(checked=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (osm_[a-z0-9_]+)\b", out))
    assert set(declared_functions()) <= exported
