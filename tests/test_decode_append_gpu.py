"""Fused decode step with cache append (VoxCPM page, "Memory & speed": one
language-model step per patch against the static cache; a full cache errors
where upstream errors)."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import assert_close_to_oracle, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import masked_gqa_attention_gb300 as M
    M.build_library()
    return M


def _step_inputs(seed, B, Hkv, D, dtype):
    g = torch.Generator().manual_seed(seed)
    kn = torch.randn((B, Hkv, 1, D), generator=g).to(dtype)
    vn = torch.randn((B, Hkv, 1, D), generator=g).to(dtype)
    return kn, vn


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_append_equals_manual_append_then_decode(M, oracle_mod, dtype):
    wl = W.static_cache_decode(seed=21, variant="span", B=4, capacity=1000, lo=100, hi=900,
                               dtype=dtype)
    B, Hq, Hkv, _, Lk, D = wl.shape
    kn, vn = _step_inputs(1, B, Hkv, D, dtype)
    q, k, v, kvl = (t.cuda() for t in (wl.q, wl.k, wl.v, wl.kv_len))
    # reference: append by hand, then the plain decode over kv_len + 1 slots
    k2, v2 = k.clone(), v.clone()
    for b in range(B):
        n = int(wl.kv_len[b])
        k2[b, :, n] = kn[b, :, 0].cuda()
        v2[b, :, n] = vn[b, :, 0].cuda()
    kvl1 = kvl + 1
    ws = M.new_decode_workspace(q, k2, v2, kv_len=kvl1)
    ref = M.masked_gqa_attn_decode(q, k2, v2, workspace=ws, scale=wl.scale, kv_len=kvl1)
    out_len = torch.zeros_like(kvl)
    out = M.masked_gqa_attn_decode_append(q, k, v, kn.cuda(), vn.cuda(), kvl, workspace=ws,
                                          kv_len_out=out_len, scale=wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(k, k2) and torch.equal(v, v2)
    assert torch.equal(out_len, kvl1)
    o_ref, _, _ = oracle_mod.attention(wl.q, k2.cpu(), v2.cpu(), scale=wl.scale,
                                       kv_len=kvl1.cpu())
    assert_close_to_oracle(out, o_ref, dtype, "append")


def test_three_steps_ping_pong_lengths(M, oracle_mod):
    wl = W.static_cache_decode(seed=33, variant="span", B=3, Hq=8, Hkv=2, D=128, capacity=600,
                               lo=10, hi=400)
    B, Hq, Hkv, _, Lk, D = wl.shape
    q, k, v = (t.cuda() for t in (wl.q, wl.k, wl.v))
    lens = [wl.kv_len.cuda(), torch.zeros_like(wl.kv_len).cuda()]
    ws = M.new_decode_workspace(q, k, v, kv_len=lens[0])
    kc, vc = wl.k.clone(), wl.v.clone()
    for step in range(3):
        kn, vn = _step_inputs(100 + step, B, Hkv, D, torch.bfloat16)
        cur, nxt = lens[step % 2], lens[(step + 1) % 2]
        n_before = cur.cpu().clone()
        out = M.masked_gqa_attn_decode_append(q, k, v, kn.cuda(), vn.cuda(), cur, workspace=ws,
                                              kv_len_out=nxt, scale=wl.scale)
        torch.cuda.synchronize()
        for b in range(B):
            kc[b, :, int(n_before[b])] = kn[b, :, 0]
            vc[b, :, int(n_before[b])] = vn[b, :, 0]
        ref, _, _ = oracle_mod.attention(wl.q, kc, vc, scale=wl.scale, kv_len=n_before + 1)
        assert_close_to_oracle(out, ref, torch.bfloat16, f"step {step}")
        assert torch.equal(nxt.cpu(), n_before + 1)


def test_full_cache_is_an_error_and_appends_nothing(M, oracle_mod):
    wl = W.static_cache_decode(seed=5, variant="span", B=2, capacity=256, lo=100, hi=200)
    B, Hq, Hkv, _, Lk, D = wl.shape
    wl.kv_len[1] = Lk  # full
    q, k, v, kvl = (t.cuda() for t in (wl.q, wl.k, wl.v, wl.kv_len))
    k0 = k.clone()
    kn, vn = _step_inputs(9, B, Hkv, D, torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_len = torch.zeros_like(kvl)
    ws = M.new_decode_workspace(q, k, v, kv_len=kvl)
    out = M.masked_gqa_attn_decode_append(q, k, v, kn.cuda(), vn.cuda(), kvl, workspace=ws,
                                          kv_len_out=out_len, scale=wl.scale, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == M.MGQA_ERR_INVALID_ARG
    assert torch.equal(k[1], k0[1])            # nothing appended to the full request
    assert int(out_len[1]) == Lk and int(out_len[0]) == int(wl.kv_len[0]) + 1
    kc = wl.k.clone()
    kc[0, :, int(wl.kv_len[0])] = kn[0, :, 0]
    vc = wl.v.clone()
    vc[0, :, int(wl.kv_len[0])] = vn[0, :, 0]
    ref, _, _ = oracle_mod.attention(wl.q, kc, vc, scale=wl.scale,
                                     kv_len=torch.tensor([int(wl.kv_len[0]) + 1, Lk]))
    assert_close_to_oracle(out, ref, torch.bfloat16, "full cache")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Hq,Hkv,D", [(16, 1, 128), (4, 4, 64), (12, 2, 64)],
                         ids=lambda v: str(v))
def test_append_head_groups_and_chunk_edges(M, oracle_mod, dtype, Hq, Hkv, D):
    """Head groups that share a KV head (16 query heads on one: two groups, one
    writer of the new row), one query head per group, and lengths at 64-slot
    chunk edges and at the cache's last slot: the new row starts a chunk no
    earlier step fetched, or fills the final slot."""
    lens = [63, 64, 127, 999]
    B, Lk = len(lens), 1000
    g, q, k, v = W.random_qkv(91 + Hq + D, B, Hq, Hkv, 1, Lk, D, dtype)
    kvl = torch.tensor(lens, dtype=torch.int32)
    kn, vn = _step_inputs(2 + D, B, Hkv, D, dtype)
    k2, v2 = k.clone(), v.clone()
    for b, n in enumerate(lens):
        k2[b, :, n] = kn[b, :, 0]
        v2[b, :, n] = vn[b, :, 0]
    qd, kd, vd, kvld = q.cuda(), k.cuda(), v.cuda(), kvl.cuda()
    out_len = torch.zeros_like(kvld)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device="cuda")
    out = M.masked_gqa_attn_decode_append(qd, kd, vd, kn.cuda(), vn.cuda(), kvld,
                                          kv_len_out=out_len, scale=D ** -0.5, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), k2) and torch.equal(vd.cpu(), v2)
    assert torch.equal(out_len.cpu(), kvl + 1)
    ref, ref_lse, _ = oracle_mod.attention(q, k2, v2, scale=D ** -0.5, kv_len=kvl + 1)
    assert_close_to_oracle(out, ref, dtype, f"append {Hq}/{Hkv}/{D}")
    assert_lse_close(lse, ref_lse, 1e-5 if dtype == torch.float32 else 1e-3)
