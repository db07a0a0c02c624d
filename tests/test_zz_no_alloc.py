"""The decode entry point without a workspace argument.

It serves callers that cannot allocate device memory for the library (a host
framework that owns every device buffer and passes an extension only its
inputs and outputs, or a per-token loop that must not touch the allocator).
The kernel's only scratch is the on-chip shared memory of its own launch.
This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

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


def _inputs(wl):
    d = {n: (getattr(wl, n).cuda() if getattr(wl, n) is not None else None)
         for n in ("q", "k", "v", "mask_bits", "kv_len", "seg_q", "seg_k")}
    return d, {n: d[n] for n in ("mask_bits", "kv_len", "seg_q", "seg_k")}


def _static_call(M, d, masks, wl):
    L = M.lib()
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
    a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, lse=lse, **masks)
    st = L.masked_gqa_attn_decode_static(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == M.MGQA_OK, L.mgqa_last_error_detail()
    return out, lse


def test_static_decode_matches_workspace_decode(M, oracle_mod):
    cases = [
        W.static_cache_decode(variant="full"),  # the 8-request, 8192-slot cache
        # one request over a long cache: several batches per CTA
        W.static_cache_decode(seed=98, variant="span", B=1, Hq=16, Hkv=2, D=64,
                              capacity=32768, lo=20000, hi=32768),
        W.static_cache_decode(seed=99, variant="span", B=5, Hq=8, Hkv=2, D=128,
                              capacity=4000, lo=10, hi=3999),  # another shape right after
        W.static_cache_decode(seed=97, variant="span", B=2, Hq=8, Hkv=1, D=128,
                              capacity=32768, lo=17000, hi=30000),
    ]
    for wl in cases:  # two calls in a row through the C ABI
        d, masks = _inputs(wl)
        ws = M.new_decode_workspace(d["q"], d["k"], d["v"], **masks)
        ref_lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
        ref = M.masked_gqa_attn_decode(d["q"], d["k"], d["v"], scale=wl.scale, workspace=ws,
                                       lse=ref_lse, **masks)
        out, lse = _static_call(M, d, masks, wl)
        torch.cuda.synchronize()
        # the same kernel with the same arithmetic: the same bits, and nothing
        # from an earlier call of another shape leaks into the result
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
        o_ref, l_ref, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
        assert_close_to_oracle(out, o_ref, torch.bfloat16, f"static decode {wl.name}")
        assert_lse_close(lse, l_ref, 1e-3)


def test_static_decode_allocates_nothing(M):
    wl = W.static_cache_decode(seed=7, variant="span", B=4, capacity=2048, lo=100, hi=2000)
    d, masks = _inputs(wl)
    out = torch.empty_like(d["q"])
    a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, **masks)
    L = M.lib()
    h = torch.cuda.current_stream().cuda_stream
    assert L.masked_gqa_attn_decode_static(ctypes.byref(a), h) == M.MGQA_OK  # warm: set-up done
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert L.masked_gqa_attn_decode_static(ctypes.byref(a), h) == M.MGQA_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_decode_has_no_size_limit(M, oracle_mod):
    # 64 requests x 32 heads: B * Hq = 2048 (no shared scratch bounds it)
    wl = W.static_cache_decode(seed=96, variant="span", B=64, Hq=32, Hkv=8, D=128,
                               capacity=256, lo=1, hi=256)
    d, masks = _inputs(wl)
    out, lse = _static_call(M, d, masks, wl)
    ref = M.masked_gqa_attn_decode(d["q"], d["k"], d["v"], scale=wl.scale, **masks)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    o_ref, l_ref, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, o_ref, torch.bfloat16, "static decode B*Hq=2048")
    assert_lse_close(lse, l_ref, 1e-3)
