"""The decode entry point that uses the library's own fixed scratch instead of
a caller-supplied workspace.

It serves callers that cannot allocate device memory for the library (a host
framework that owns every device buffer and passes an extension only its
inputs and outputs, or a per-token loop that must not touch the allocator).
This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads as W
from _util import BF16_MAX_ABS, BF16_MEAN_ABS

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


def _close(a, b):
    err = (a.double() - b.double()).abs()
    return err.max().item() <= BF16_MAX_ABS and err.mean().item() <= BF16_MEAN_ABS


def test_static_scratch_decode_matches_workspace_decode(M):
    L = M.lib()
    stream = torch.cuda.current_stream()
    cases = [
        W.static_cache_decode(variant="full"),  # the 8-request, 8192-slot cache
        W.static_cache_decode(seed=99, variant="span", B=5, Hq=8, Hkv=2, D=128,
                              capacity=4000, lo=10, hi=3999),  # another shape right after
    ]
    for wl in cases:  # two calls in a row through the C ABI
        d, masks = _inputs(wl)
        ref = M.masked_gqa_attn_decode(d["q"], d["k"], d["v"], scale=wl.scale,
                                       workspace=M.new_decode_workspace(d["q"], d["k"], d["v"], **masks),
                                       **masks)
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
        a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, lse=lse, **masks)
        st = L.masked_gqa_attn_decode_static(ctypes.byref(a), stream.cuda_stream)
        assert st == M.MGQA_OK, L.mgqa_last_error_detail()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert _close(out, ref)


def test_static_scratch_rejects_oversized_calls(M):
    L = M.lib()
    # 64 requests x 32 heads x 32768 slots need far more than the fixed scratch
    # (the cache is a broadcast view: the call is rejected before any launch)
    q = torch.zeros((64, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((64, 8, 1, 128), dtype=torch.bfloat16, device="cuda").expand(64, 8, 32768, 128)
    a = M.make_args(q, k, k, q.clone())
    need = L.masked_gqa_attn_decode_workspace_size(ctypes.byref(a))
    assert need > M.DECODE_STATIC_SCRATCH_BYTES
    st = L.masked_gqa_attn_decode_static(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == M.MGQA_ERR_UNSUPPORTED
    assert b"scratch" in L.mgqa_last_error_detail()
