"""Parity of the static-cache decode kernel against the fp64 oracle, plus the
page invariants it must keep bit for bit: masked slots add exact zeros
(VoxCPM page, "Upstream-identical practice", attention bullet) and the
filled-span form equals the full-cache form (VoxCPM page, "Memory & speed",
attention_span paragraph)."""
import numpy as np
import pytest
import torch

import workloads as W
from _util import assert_close_to_oracle, assert_lse_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import masked_gqa_attention_gb300 as M
    M.build_library()
    return M


def run_decode(M, wl, ws=None, lse=True, err=None):
    d = to_device(wl)
    out = torch.empty_like(d["q"])
    lse_t = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda") if lse else None
    masks = {k: d[k] for k in ("mask_bits", "kv_len", "seg_q", "seg_k")}
    M.masked_gqa_attn_decode(d["q"], d["k"], d["v"], out, workspace=ws, scale=wl.scale,
                             lse=lse_t, dev_error=err, **masks)
    torch.cuda.synchronize()
    return out, lse_t, ws


@pytest.mark.parametrize("variant", ["full", "span"])
def test_static_cache_decode_matches_oracle(M, oracle_mod, variant):
    wl = W.static_cache_decode(variant=variant)
    out, lse, _ = run_decode(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, torch.bfloat16, f"decode {variant}")
    assert_lse_close(lse, ref_lse, 1e-3)


def test_full_cache_and_filled_span_are_bit_identical(M):
    full = W.static_cache_decode(variant="full")
    span = W.static_cache_decode(variant="span")
    assert torch.equal(full.k, span.k)
    o1, l1, _ = run_decode(M, full)
    o2, l2, _ = run_decode(M, span)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_masked_slots_refill_leaves_bits(M):
    wl = W.static_cache_decode(variant="span")
    o1, l1, ws = run_decode(M, wl)
    g = torch.Generator().manual_seed(123)
    for b, n in enumerate(wl.info["filled"]):
        wl.k[b, :, n:] = (torch.randn(wl.k[b, :, n:].shape, generator=g) * 3e4).to(wl.k.dtype)
        wl.v[b, :, n:] = float("nan")  # never read: masked slots are not fetched
    o2, l2, _ = run_decode(M, wl, ws=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_repeated_calls_same_bits_workspace_untouched(M):
    # the splits merge on chip: a workspace passed in is never read or
    # written, and repeated calls give the same bits with or without one
    wl = W.static_cache_decode(variant="full", seed=4242)
    o1, l1, _ = run_decode(M, wl)
    ws = torch.full((1 << 16,), 0xAB, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        o2, l2, _ = run_decode(M, wl, ws=ws)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert bool(torch.all(ws == 0xAB))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("Hq,Hkv,D", [(16, 2, 64), (8, 8, 128), (12, 2, 64), (16, 1, 128), (4, 2, 128)])
@pytest.mark.parametrize("Lk", [8192, 300, 129, 1])
def test_decode_shapes_and_dtypes(M, oracle_mod, dtype, Hq, Hkv, D, Lk):
    lo = 0 if Lk < 40 else 1
    wl = W.static_cache_decode(seed=Lk + Hq + D, variant="span", B=3, Hq=Hq, Hkv=Hkv, D=D,
                               capacity=Lk, lo=lo, hi=Lk, dtype=dtype)
    out, lse, _ = run_decode(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, dtype, f"decode {Hq}/{Hkv}/{D}/{Lk}")
    assert_lse_close(lse, ref_lse, 1e-5 if dtype == torch.float32 else 1e-3)


def test_decode_empty_and_holey_masks(M, oracle_mod):
    B, Hq, Hkv, Lk, D = 4, 8, 2, 1000, 64
    g, q, k, v = W.random_qkv(7, B, Hq, Hkv, 1, Lk, D, torch.bfloat16)
    m = torch.rand((B, 1, Lk), generator=g) < 0.3
    m[0] = False                # a request with nothing to attend to
    m[1, :, 200:] = False       # a prefix
    m[2, :, :900] = False       # a suffix inside the last chunk
    wl = W.Workload("holes", q, k, v, 0.125, mask_bits=W.pack_bool_mask(m))
    wl.kv_len = torch.tensor([Lk, 600, Lk, 33], dtype=torch.int32)
    out, lse, _ = run_decode(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, torch.bfloat16, "decode holes")
    assert_lse_close(lse, ref_lse, 1e-3)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_segment_ids(M, oracle_mod):
    B, Hq, Hkv, Lk, D = 2, 4, 1, 777, 128
    g, q, k, v = W.random_qkv(17, B, Hq, Hkv, 1, Lk, D, torch.bfloat16)
    seg_k = (torch.arange(Lk) // 100).to(torch.int32).repeat(B, 1).contiguous()
    seg_q = torch.tensor([[3], [7]], dtype=torch.int32)
    wl = W.Workload("seg", q, k, v, 0.09, seg_q=seg_q, seg_k=seg_k)
    out, lse, _ = run_decode(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, torch.bfloat16, "decode seg")


def test_cache_full_is_reported_and_clamped(M, oracle_mod):
    wl = W.static_cache_decode(seed=5, variant="span", B=2, capacity=512, lo=100, hi=400)
    wl.kv_len[1] = 600  # more than the cache holds
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = run_decode(M, wl, err=err)
    assert int(err.item()) == M.MGQA_ERR_INVALID_ARG
    wl.kv_len[1] = 512
    ref, _, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, torch.bfloat16, "decode clamped")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("B,Hq,Hkv,D", [(1, 16, 2, 64), (2, 8, 1, 128), (1, 4, 4, 64)])
def test_long_cache_many_batches(M, oracle_mod, dtype, B, Hq, Hkv, D):
    """A 32768-slot cache filled past 17000 slots: every CTA runs several
    batches of rows (the running maximum carried from batch to batch); the
    bitmask and filled-length forms stay bit-identical."""
    wl = W.static_cache_decode(seed=B + Hq + D, variant="span", B=B, Hq=Hq, Hkv=Hkv, D=D,
                               capacity=32768, lo=17000, hi=32768, dtype=dtype)
    out, lse, _ = run_decode(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, dtype, f"long cache {B}/{Hq}/{Hkv}/{D}")
    assert_lse_close(lse, ref_lse, 1e-5 if dtype == torch.float32 else 1e-3)
    full = W.static_cache_decode(seed=B + Hq + D, variant="full", B=B, Hq=Hq, Hkv=Hkv, D=D,
                                 capacity=32768, lo=17000, hi=32768, dtype=dtype)
    o2, l2, _ = run_decode(M, full)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_shapes_back_to_back(M, oracle_mod):
    """Calls of different shapes (cluster grids of different sizes) in a row:
    no state carries from one call to the next."""
    shapes = [dict(B=1, Hq=16, Hkv=2, D=64, capacity=32768, lo=20000, hi=32768),
              dict(B=2, Hq=8, Hkv=1, D=128, capacity=32768, lo=17000, hi=30000),
              dict(B=8, Hq=16, Hkv=2, D=64, capacity=8192, lo=256, hi=3100),
              dict(B=3, Hq=4, Hkv=4, D=128, capacity=5000, lo=1, hi=5000)]
    for i, kw in enumerate(shapes * 2):
        wl = W.static_cache_decode(seed=300 + i, variant="span", **kw)
        out, lse, _ = run_decode(M, wl)
        ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
        assert_close_to_oracle(out, ref, torch.bfloat16, f"shape {i}")
        assert_lse_close(lse, ref_lse, 1e-3)
