"""Packed-guidance helpers (OmniVoice page, "Memory & speed", packed_guidance):
pack a conditional and an unconditional sequence into one block-diagonal row,
attend, and split the output back; each block equals its sequence run alone."""
import pytest
import torch

import workloads as W
from _util import assert_close_to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import masked_gqa_attention_gb300 as M
    M.build_library()
    return M


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_pack_unpack_roundtrip(M, dtype):
    g = torch.Generator().manual_seed(4)
    a = torch.randn((2, 8, 1024, 128), generator=g).to(dtype).cuda()
    b = torch.randn((2, 8, 384, 128), generator=g).to(dtype).cuda()
    packed, seg = M.masked_gqa_pack_pair(a, b)
    torch.cuda.synchronize()
    assert torch.equal(packed, torch.cat([a, b], dim=2))
    assert torch.equal(seg.cpu(), torch.cat([torch.zeros(2, 1024), torch.ones(2, 384)], 1).int())
    a2, b2 = M.masked_gqa_unpack_pair(packed, 1024)
    torch.cuda.synchronize()
    assert torch.equal(a2, a) and torch.equal(b2, b)


def test_packed_guidance_end_to_end(M, oracle_mod):
    """cond (1024) and uncond target (384) packed, attended, unpacked: each
    half matches the oracle of its sequence alone."""
    Hq, Hkv, D = 16, 8, 128
    gc, qc, kc, vc = W.random_qkv(11, 1, Hq, Hkv, 1024, 1024, D, torch.bfloat16)
    gu, qu, ku, vu = W.random_qkv(12, 1, Hq, Hkv, 384, 384, D, torch.bfloat16)
    qp, seg = M.masked_gqa_pack_pair(qc.cuda(), qu.cuda())
    kp, _ = M.masked_gqa_pack_pair(kc.cuda(), ku.cuda())
    vp, _ = M.masked_gqa_pack_pair(vc.cuda(), vu.cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = M.masked_gqa_attn_prefill(qp, kp, vp, scale=D ** -0.5, seg_q=seg, seg_k=seg,
                                    dev_error=err)
    oc, ou = M.masked_gqa_unpack_pair(out, 1024)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "a bounded wait gave up"
    rc, _, _ = oracle_mod.attention(qc, kc, vc, scale=D ** -0.5)
    ru, _, _ = oracle_mod.attention(qu, ku, vu, scale=D ** -0.5)
    assert_close_to_oracle(oc, rc, torch.bfloat16, "cond block")
    assert_close_to_oracle(ou, ru, torch.bfloat16, "uncond block")
