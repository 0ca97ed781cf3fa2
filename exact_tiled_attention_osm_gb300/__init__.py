"""Python binding of libosm, the C-ABI library of exact online-softmax attention.

Argument marshalling only: every step of every operation runs in the CUDA
kernels of libosm.so.  PyTorch provides device memory and the current CUDA
stream.  There is no CPU fallback: if the library is missing or fails to load,
every call raises.

Functions mirror the C entry points in include/osm.h:
    softmax_rows(x, out=None)                          -> y
    softmax_topk(x, k, idx=None, prob=None)            -> (idx, prob)
    attn_fwd(q, k, v, scale=None, causal=False, key_len=None, out=None, lse=None,
             score_bound=None)                         -> (o, lse)
    attn_bwd(q, k, v, o, lse, dout, scale=None, causal=False, key_len=None,
             workspace=None)                           -> (dq, dk, dv)
    attn_bwd_workspace_bytes(B, H, Nq)                  -> int
    attn_decode_splitkv(q, k, v, scale=None, key_len=None, num_splits=16,
                        workspace=None, out=None, lse=None) -> (o, lse)
    attn_decode_splitkv_noalloc(q, k, v, scale=None, key_len=None, num_splits=16,
                                out=None, lse=None)     -> (o, lse)
    decode_workspace_bytes(B, H, d, num_splits)         -> int
    decode_partials(workspace, B, H, d, num_splits)     -> (m, l, o~) views
    decode_state(B, H, d, device)                       -> (m, l, o~), the empty summary
    decode_append_workspace_bytes(B, H, d, num_splits)  -> int
    attn_decode_append(q, k, v, state, key_start=None, key_end=None, scale=None,
                       num_splits=16, workspace=None, out=None, lse=None) -> (o, lse)
    lse_merge(o_parts, lse_parts, out_dtype=torch.float32) -> (o, lse)
    selftest_bounded_wait(device=None)                  (runs a wait that must give up)
    device_status()                                    -> int (0 = no device wait ran out)
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libosm.so")

(OSM_OK, OSM_ERR_INVALID_VALUE, OSM_ERR_UNSUPPORTED, OSM_ERR_CUDA, OSM_ERR_TIMEOUT,
 OSM_ERR_CONFLICT, OSM_ERR_INDEX) = range(7)
OSM_F32, OSM_BF16 = 0, 1

# exported names and their C signatures (include/osm.h)
_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "osm_softmax_rows": (_I, [_P, _P, _I64, _I64, _P]),
    "osm_softmax_topk": (_I, [_P, _I64, _I64, _I, _P, _P, _P]),
    "osm_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P]),
    "osm_attn_fwd_bounded": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _F, _P]),
    "osm_attn_fwd_normalised": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P]),
    "osm_attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "osm_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P,
                          _SZ, _P]),
    "osm_attn_decode_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "osm_attn_decode_splitkv": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _I, _P, _SZ, _P]),
    "osm_attn_decode_splitkv_noalloc": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _I, _P]),
    "osm_attn_decode_append_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "osm_attn_decode_append": (_I, [_I, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P,
                                    _P, _I, _P, _SZ, _P]),
    "osm_lse_merge": (_I, [_P, _P, _I, _I64, _I, _I, _P, _P, _P]),
    "osm_status_string": (ctypes.c_char_p, [_I]),
    "osm_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "osm_selftest_bounded_wait": (_I, [_P]),
    "osm_abi_version": (_I, []),
}

_lib = None


class OsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libosm.so (building it first with nvcc if it is not there)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        from . import build as _build
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().osm_status_string(int(status)).decode()


def _check(st: int, where: str):
    if st != OSM_OK:
        raise OsmError(st, where)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype=None, device=None, shape=None):
    """Check what the C entry points cannot: a contiguous CUDA tensor of the
    given dtype, device and shape (a short output buffer would be overrun)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libosm has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def softmax_rows(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Row softmax of a [rows, cols] fp32 CUDA tensor (out may be x for in place)."""
    _need(x, "x", torch.float32)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    y = torch.empty_like(x) if out is None else out
    _need(y, "out", torch.float32, x.device, x.shape)
    if y.shape != x.shape:
        raise ValueError("out must have x's shape")
    lib = load_library()
    with torch.cuda.device(x.device):
        _check(lib.osm_softmax_rows(x.data_ptr(), y.data_ptr(), x.shape[0], x.shape[1],
                                    _stream(x)), "osm_softmax_rows")
    return y


def softmax_topk(x, k, idx=None, prob=None):
    """Top-k of every row of x ([rows, cols] fp32 CUDA) with softmax probabilities.

    Returns (idx [rows, k] int32, prob [rows, k] fp32): larger value first,
    ties by smaller column.
    """
    _need(x, "x", torch.float32)
    if x.dim() != 2:
        raise ValueError("x must be [rows, cols]")
    rows, cols = x.shape
    idx_t = torch.empty((rows, k), dtype=torch.int32, device=x.device) if idx is None else idx
    prob_t = torch.empty((rows, k), dtype=torch.float32, device=x.device) if prob is None else prob
    _need(idx_t, "idx", torch.int32, x.device, (rows, k))
    _need(prob_t, "prob", torch.float32, x.device, (rows, k))
    lib = load_library()
    with torch.cuda.device(x.device):
        _check(lib.osm_softmax_topk(x.data_ptr(), rows, cols, int(k), idx_t.data_ptr(),
                                    prob_t.data_ptr(), _stream(x)), "osm_softmax_topk")
    return idx_t, prob_t


def attn_fwd(q, k, v, scale=None, causal=False, key_len=None, out=None, lse=None,
             score_bound=None, normalised=False):
    """Attention forward.  q [B,H,Nq,d], k, v [B,H,Nk,d] bf16 CUDA; key_len int32 [B] or None.

    Returns (o [B,H,Nq,d] bf16, lse [B,H,Nq] fp32).  `score_bound`: a known
    upper bound on the scaled scores (osm_attn_fwd_bounded); None = unknown.
    `normalised`: compute the normalised form, dividing by l after every key
    tile (osm_attn_fwd_normalised; not with a score bound).
    """
    if normalised and score_bound is not None:
        raise ValueError("normalised form takes no score bound")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, q.device)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,H,Nq,d] and k, v [B,H,Nk,d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q, k, v disagree on B, H or d")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "out", torch.bfloat16, q.device, q.shape)
    _need(lse_t, "lse", torch.float32, q.device, (B, H, Nq))
    kl = 0
    if key_len is not None:
        _need(key_len, "key_len", torch.int32, q.device, (B,))
        kl = key_len.data_ptr()
    lib = load_library()
    with torch.cuda.device(q.device):
        if normalised:
            _check(lib.osm_attn_fwd_normalised(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse_t.data_ptr(), B, H, Nq, Nk, d,
                                               float(scale), int(bool(causal)), kl, _stream(q)),
                   "osm_attn_fwd_normalised")
        elif score_bound is None:
            _check(lib.osm_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse_t.data_ptr(), B, H, Nq, Nk, d, float(scale),
                                    int(bool(causal)), kl, _stream(q)), "osm_attn_fwd")
        else:
            _check(lib.osm_attn_fwd_bounded(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse_t.data_ptr(), B, H, Nq, Nk, d,
                                            float(scale), int(bool(causal)), kl,
                                            float(score_bound), _stream(q)),
                   "osm_attn_fwd_bounded")
    return o, lse_t


def attn_bwd_workspace_bytes(B: int, H: int, Nq: int) -> int:
    return int(load_library().osm_attn_bwd_workspace_bytes(B, H, Nq))


def attn_bwd(q, k, v, o, lse, dout, scale=None, causal=False, key_len=None, workspace=None):
    """Gradients of attention.  q, o, dout [B,H,Nq,d]; k, v [B,H,Nk,d] bf16 CUDA;
    lse [B,H,Nq] fp32 (from attn_fwd).  Returns (dq, dk, dv), bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n, torch.bfloat16, q.device)
    _need(lse, "lse", torch.float32, q.device)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape or o.shape != q.shape \
            or dout.shape != q.shape or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("shapes: q, o, dout [B,H,Nq,d]; k, v [B,H,Nk,d]; lse [B,H,Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    need = int(lib.osm_attn_bwd_workspace_bytes(B, H, Nq))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    kl = 0
    if key_len is not None:
        _need(key_len, "key_len", torch.int32, q.device, (B,))
        kl = key_len.data_ptr()
    with torch.cuda.device(q.device):
        _check(lib.osm_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                                kl, workspace.data_ptr(), workspace.numel(), _stream(q)),
               "osm_attn_bwd")
    return dq, dk, dv


def decode_workspace_bytes(B: int, H: int, d: int, num_splits: int) -> int:
    return int(load_library().osm_attn_decode_splitkv_workspace_bytes(B, H, d, num_splits))


def attn_decode_splitkv(q, k, v, scale=None, key_len=None, num_splits=16, workspace=None,
                        out=None, lse=None):
    """Split-KV decode.  q [B,H,1,d], k, v [B,H,Nk,d] (bf16 or fp32, same dtype).

    Returns (o [B,H,1,d], lse [B,H]).  `workspace` (uint8 CUDA tensor) keeps the
    per-split (m, l, o~) summaries in the layout documented in osm.h.
    """
    dt = {torch.bfloat16: OSM_BF16, torch.float32: OSM_F32}.get(q.dtype)
    if dt is None:
        raise ValueError("decode supports bf16 and fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, one, d = q.shape
    if one != 1 or k.dim() != 4 or v.shape != k.shape or k.shape[0] != B or k.shape[1] != H \
            or k.shape[3] != d:
        raise ValueError("q must be [B,H,1,d] and k, v [B,H,Nk,d]")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = decode_workspace_bytes(B, H, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, q.device)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "out", q.dtype, q.device, q.shape)
    _need(lse_t, "lse", torch.float32, q.device, (B, H))
    kl = 0
    if key_len is not None:
        _need(key_len, "key_len", torch.int32, q.device, (B,))
        kl = key_len.data_ptr()
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.osm_attn_decode_splitkv(dt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           o.data_ptr(), lse_t.data_ptr(), B, H, Nk, d,
                                           float(scale), kl, int(num_splits),
                                           workspace.data_ptr(), workspace.numel(), _stream(q)),
               "osm_attn_decode_splitkv")
    return o, lse_t


def decode_append_workspace_bytes(B: int, H: int, d: int, num_splits: int) -> int:
    return int(load_library().osm_attn_decode_append_workspace_bytes(B, H, d, num_splits))


def decode_state(B: int, H: int, d: int, device) -> tuple:
    """The empty running summary (m = -inf, l = 0, o~ = 0) for attn_decode_append."""
    return (torch.full((B, H), -math.inf, dtype=torch.float32, device=device),
            torch.zeros((B, H), dtype=torch.float32, device=device),
            torch.zeros((B, H, d), dtype=torch.float32, device=device))


def attn_decode_append(q, k, v, state, key_start=None, key_end=None, scale=None,
                       num_splits=16, workspace=None, out=None, lse=None):
    """Extend each query's running summary by the keys [key_start[b], key_end[b]).

    q [B,H,1,d]; k, v [B,H,Nk,d] (bf16 or fp32, same dtype); state = (m [B,H],
    l [B,H], o~ [B,H,d]) fp32 CUDA tensors, updated in place.  Returns (o, lse),
    the attention output over every key merged into the state so far.
    """
    dt = {torch.bfloat16: OSM_BF16, torch.float32: OSM_F32}.get(q.dtype)
    if dt is None:
        raise ValueError("decode supports bf16 and fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, one, d = q.shape
    if one != 1 or k.dim() != 4 or v.shape != k.shape or k.shape[0] != B or k.shape[1] != H \
            or k.shape[3] != d:
        raise ValueError("q must be [B,H,1,d] and k, v [B,H,Nk,d]")
    Nk = k.shape[2]
    sm, sl, so = state
    for t, n, shp in ((sm, "state m", (B, H)), (sl, "state l", (B, H)), (so, "state o", (B, H, d))):
        _need(t, n, torch.float32, q.device)
        if tuple(t.shape) != shp:
            raise ValueError(f"{n} must have shape {shp}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = decode_append_workspace_bytes(B, H, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, q.device)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "out", q.dtype, q.device, q.shape)
    _need(lse_t, "lse", torch.float32, q.device, (B, H))
    ptrs = []
    for t, n in ((key_start, "key_start"), (key_end, "key_end")):
        if t is None:
            ptrs.append(0)
        else:
            _need(t, n, torch.int32, q.device, (B,))
            ptrs.append(t.data_ptr())
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.osm_attn_decode_append(dt, q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, Nk,
                                          d, float(scale), ptrs[0], ptrs[1], sm.data_ptr(),
                                          sl.data_ptr(), so.data_ptr(), o.data_ptr(),
                                          lse_t.data_ptr(), int(num_splits),
                                          workspace.data_ptr(), workspace.numel(), _stream(q)),
               "osm_attn_decode_append")
    return o, lse_t


# bytes of the library's own scratch area used by attn_decode_splitkv_noalloc
NOALLOC_SCRATCH_BYTES = 32 << 20


def attn_decode_splitkv_noalloc(q, k, v, scale=None, key_len=None, num_splits=16, out=None,
                                lse=None):
    """Split-KV decode that allocates nothing on the device inside the library.

    For callers that cannot allocate device memory (for example a plug-in whose
    host program owns all device memory): the split summaries live in a fixed
    scratch area of NOALLOC_SCRATCH_BYTES inside libosm, shared by every call on
    the device, so calls must not overlap on the GPU.  Output tensors are
    allocated here only when `out` / `lse` are not given.
    """
    dt = {torch.bfloat16: OSM_BF16, torch.float32: OSM_F32}.get(q.dtype)
    if dt is None:
        raise ValueError("decode supports bf16 and fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, one, d = q.shape
    if one != 1 or k.dim() != 4 or v.shape != k.shape or k.shape[0] != B or k.shape[1] != H \
            or k.shape[3] != d:
        raise ValueError("q must be [B,H,1,d] and k, v [B,H,Nk,d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "out", q.dtype, q.device, q.shape)
    _need(lse_t, "lse", torch.float32, q.device, (B, H))
    kl = 0
    if key_len is not None:
        _need(key_len, "key_len", torch.int32, q.device, (B,))
        kl = key_len.data_ptr()
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.osm_attn_decode_splitkv_noalloc(dt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                   o.data_ptr(), lse_t.data_ptr(), B, H,
                                                   k.shape[2], d, float(scale), kl,
                                                   int(num_splits), _stream(q)),
               "osm_attn_decode_splitkv_noalloc")
    return o, lse_t


def decode_partials(workspace: torch.Tensor, B: int, H: int, d: int, num_splits: int):
    """Views (m [S,B*H], l [S,B*H], o~ [S,B*H,d]) of a decode workspace (layout in osm.h)."""
    n = num_splits * B * H
    a = ((n * 4 + 255) // 256) * 256
    f = workspace.view(torch.uint8)
    m = f[:n * 4].view(torch.float32).view(num_splits, B * H)
    l = f[a:a + n * 4].view(torch.float32).view(num_splits, B * H)
    o = f[2 * a:2 * a + n * d * 4].view(torch.float32).view(num_splits, B * H, d)
    return m, l, o


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out_dtype=torch.float32):
    """Merge normalised partials: o_parts [S, rows, d] fp32, lse_parts [S, rows] fp32."""
    _need(o_parts, "o_parts", torch.float32)
    _need(lse_parts, "lse_parts", torch.float32, o_parts.device)
    S, rows, d = o_parts.shape
    if lse_parts.shape != (S, rows):
        raise ValueError("lse_parts must be [S, rows]")
    odt = {torch.bfloat16: OSM_BF16, torch.float32: OSM_F32}[out_dtype]
    o = torch.empty((rows, d), dtype=out_dtype, device=o_parts.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    lib = load_library()
    with torch.cuda.device(o_parts.device):
        _check(lib.osm_lse_merge(o_parts.data_ptr(), lse_parts.data_ptr(), S, rows, d, odt,
                                 o.data_ptr(), lse.data_ptr(), _stream(o_parts)), "osm_lse_merge")
    return o, lse


def selftest_bounded_wait(device=None) -> None:
    """Launch the bounded-wait self-test (a wait that runs out; see osm.h)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.osm_selftest_bounded_wait(torch.cuda.current_stream(dev).cuda_stream),
               "osm_selftest_bounded_wait")


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    lib = load_library()
    w = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib.osm_device_status(torch.cuda.current_stream(dev).cuda_stream, ctypes.byref(w))
    if st not in (OSM_OK, OSM_ERR_TIMEOUT, OSM_ERR_CONFLICT, OSM_ERR_INDEX):
        raise OsmError(st, "osm_device_status")
    return int(w.value)
