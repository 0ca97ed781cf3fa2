"""The Python binding refuses, before any launch, tensors the C entry points
cannot check: a short output buffer would be written past its end."""
import pytest
import torch

import exact_tiled_attention_osm_gb300 as osm

pytestmark = pytest.mark.gpu


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16, device="cuda")


def f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32, device="cuda")


def test_short_outputs_are_refused(cuda_ok):
    q, k = bf16(2, 3, 130, 128), bf16(2, 3, 200, 128)
    with pytest.raises(ValueError):
        osm.attn_fwd(q, k, k, out=bf16(2, 3, 129, 128))
    with pytest.raises(ValueError):
        osm.attn_fwd(q, k, k, lse=f32(2, 3, 129))
    with pytest.raises(ValueError):
        osm.attn_fwd(q, k, k, key_len=torch.full((3,), 5, dtype=torch.int32, device="cuda"))
    x = f32(4, 1000)
    with pytest.raises(ValueError):
        osm.softmax_rows(x, out=f32(4, 999))
    with pytest.raises(ValueError):
        osm.softmax_topk(x, 8, idx=torch.zeros(4, 7, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        osm.softmax_topk(x, 8, prob=f32(3, 8))
    qd, kd = bf16(2, 3, 1, 64), bf16(2, 3, 500, 64)
    with pytest.raises(ValueError):
        osm.attn_decode_splitkv(qd, kd, kd, out=bf16(2, 2, 1, 64))
    with pytest.raises(ValueError):
        osm.attn_decode_splitkv(qd, kd, kd, lse=f32(2))
    with pytest.raises(ValueError):
        osm.attn_decode_splitkv(qd, kd, kd, out=f32(2, 3, 1, 64))  # wrong dtype
    with pytest.raises(ValueError):
        osm.attn_decode_splitkv_noalloc(qd, kd, kd, lse=f32(2, 2))
    state = osm.decode_state(2, 3, 64, "cuda")
    with pytest.raises(ValueError):
        osm.attn_decode_append(qd, kd, kd, state,
                               key_end=torch.full((1,), 5, dtype=torch.int32, device="cuda"))
    # nothing was launched, so nothing ran out
    assert osm.device_status() == 0


def test_well_formed_outputs_are_used_in_place(cuda_ok):
    q = torch.randn(1, 2, 64, 128, device="cuda").to(torch.bfloat16)
    o, lse = bf16(1, 2, 64, 128), f32(1, 2, 64)
    o2, lse2 = osm.attn_fwd(q, q, q, out=o, lse=lse)
    assert o2.data_ptr() == o.data_ptr() and lse2.data_ptr() == lse.data_ptr()
    assert torch.isfinite(lse).all()
