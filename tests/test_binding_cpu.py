"""The Python binding marshals only: with host tensors (no GPU here) every
entry point refuses before anything reaches the library, so there is no
silent CPU path; wrongly typed side inputs are refused the same way."""
import pytest
import torch

import masked_gqa_attention_gb300 as M


def _qkv(Lq=8, Lk=8, D=64, dtype=torch.bfloat16):
    q = torch.zeros(1, 4, Lq, D, dtype=dtype)
    k = torch.zeros(1, 2, Lk, D, dtype=dtype)
    return q, k, k.clone()


def test_prefill_refuses_host_tensors():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_attn_prefill(q, k, v, scale=0.125)


def test_decode_entry_points_refuse_host_tensors():
    q, k, v = _qkv(Lq=1)
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_attn_decode(q, k, v, workspace=torch.zeros(16, dtype=torch.uint8), scale=0.125)
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_attn_decode_static(q, k, v, scale=0.125)
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_attn_decode_append(q, k, v, k[:, :, :1], v[:, :, :1],
                                        torch.zeros(1, dtype=torch.int32),
                                        workspace=torch.zeros(16, dtype=torch.uint8), scale=0.125)


def test_pack_and_rope_refuse_host_tensors():
    q, k, _ = _qkv()
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_pack_pair(q, q)
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_unpack_pair(q, 4)
    with pytest.raises(ValueError, match="CUDA"):
        M.masked_gqa_rope(q, torch.ones(32, dtype=torch.float32))


def test_every_exported_entry_point_has_a_binding():
    for name in M.EXPORTED_SYMBOLS:
        if name.startswith("masked_gqa"):
            assert callable(getattr(M, name)), name
