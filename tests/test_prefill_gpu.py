"""Parity of the prefill kernels against the fp64 oracle on the engine pages'
workload shapes and on seeded ragged cases, plus the invariants the pages
state: masked keys add exact zeros, a packed block-diagonal row equals each
block run alone, grouped KV heads equal explicitly repeated heads."""
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


def run_prefill(M, wl, lse=True, err=None, d=None):
    """Every call carries a device error flag, so a bounded wait that gave up
    (which would leave stale output behind) fails the test by itself."""
    d = d or to_device(wl)
    out = torch.full_like(d["q"], float("nan"))
    lse_t = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda") if lse else None
    own = err is None
    if own:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.masked_gqa_attn_prefill(d["q"], d["k"], d["v"], out, scale=wl.scale, lse=lse_t,
                              dev_error=err, mask_bits=d["mask_bits"], kv_len=d["kv_len"],
                              seg_q=d["seg_q"], seg_k=d["seg_k"], causal=wl.causal)
    torch.cuda.synchronize()
    if own:
        assert int(err.item()) == 0, f"device error {int(err.item())}"
    return out, lse_t


def oracle(oracle_mod, wl, rows=None):
    q, k, v, masks = wl.q, wl.k, wl.v, wl.masks()
    if rows is not None:
        q, k, v = q[rows], k[rows], v[rows]
        masks = {n: (t[rows] if t is not None else None) for n, t in masks.items()}
    out, lse, _ = oracle_mod.attention(q, k, v, scale=wl.scale, **masks)
    return out, lse


def test_tiny_fp32_config(M, oracle_mod):
    wl = W.tiny_fp32()
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.float32, "tiny fp32")
    assert_lse_close(lse, ref_lse, 1e-5)


@pytest.mark.parametrize("variant", ["bits", "kvlen"])
def test_padded_cfg_config(M, oracle_mod, variant):
    wl = W.padded_cfg(variant=variant)
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.bfloat16, f"padded cfg {variant}")
    assert_lse_close(lse, ref_lse, 2e-3)


def test_padded_cfg_broadcast_key_padding_mask(M, oracle_mod):
    """The key-padding mask as one row of words per batch row ([B, 1, W],
    query stride 0; OmniVoice page, "Upstream-identical practice", attention-
    mask bullet) gives the oracle's result and the full 4D mask's bits."""
    wl = W.padded_cfg(variant="bits")
    full_out, full_lse = run_prefill(M, wl)
    wl.mask_bits = wl.mask_bits[:, :1, :].contiguous()  # [2, 1, 32]: 128 B per batch row
    d = to_device(wl)
    out, lse = run_prefill(M, wl, d=d)
    assert torch.equal(out, full_out) and torch.equal(lse, full_lse)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale,
                                           mask_bits=wl.mask_bits.expand(2, 1024, 32))
    assert_close_to_oracle(out, ref, torch.bfloat16, "broadcast key padding")
    assert_lse_close(lse, ref_lse, 2e-3)


def test_broadcast_mask_over_batch_and_queries(M, oracle_mod):
    """One mask row for every batch row and query (both strides 0), with holes."""
    wl = W.random_case(12, 3, 4, 2, 300, 450, 128, dtype=torch.bfloat16, mask="bits")
    row = wl.mask_bits[1:2, 5:6, :].contiguous()  # [1, 1, W]
    wl.mask_bits = row
    out, lse = run_prefill(M, wl)
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale,
                                           mask_bits=row.expand(3, 300, row.shape[2]))
    assert_close_to_oracle(out, ref, torch.bfloat16, "broadcast over batch and queries")
    assert_lse_close(lse, ref_lse, 2e-3)


def test_padded_cfg_bits_equal_kvlen_bitwise(M):
    o1, l1 = run_prefill(M, W.padded_cfg(variant="bits"))
    o2, l2 = run_prefill(M, W.padded_cfg(variant="kvlen"))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_padded_cfg_masked_keys_refill(M):
    wl = W.padded_cfg(variant="bits")
    o1, l1 = run_prefill(M, wl)
    g = torch.Generator().manual_seed(3)
    wl.k[1, :, 384:] = (torch.randn(wl.k[1, :, 384:].shape, generator=g) * 50).to(torch.bfloat16)
    wl.v[1, :, 384:] = (torch.randn(wl.v[1, :, 384:].shape, generator=g) * 1e4).to(torch.bfloat16)
    o2, l2 = run_prefill(M, wl)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_packed_guidance_config_and_blocks_alone(M, oracle_mod):
    wl = W.packed_guidance()
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.bfloat16, "packed")
    assert_lse_close(lse, ref_lse, 2e-3)
    for lo, hi in wl.info["segments"]:
        alone = W.Workload("alone", wl.q[:, :, lo:hi].contiguous(), wl.k[:, :, lo:hi].contiguous(),
                           wl.v[:, :, lo:hi].contiguous(), wl.scale)
        o2, l2 = run_prefill(M, alone)
        # block boundaries fall on 128-row tiles here, so the bits agree exactly
        assert torch.equal(out[:, :, lo:hi], o2) and torch.equal(lse[:, :, lo:hi], l2)


def test_missed_speculation_repeated(M):
    """Query tiles of the second packed block find key tile 0 empty, so the
    speculative first load misses and stage 0 runs one phase late. Repeated
    back-to-back launches (no host sync in between) vary the timing between
    the producer and the MMA warp: no wait may give up and every run must
    give the same bits as a run after a full synchronisation."""
    wl = W.packed_guidance()
    d = to_device(wl)
    ref, _ = run_prefill(M, wl, lse=False, d=d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(24):
        o = torch.empty_like(d["q"])
        M.masked_gqa_attn_prefill(d["q"], d["k"], d["v"], o, scale=wl.scale, dev_error=err,
                                  seg_q=d["seg_q"], seg_k=d["seg_k"])
        outs.append(o)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for o in outs:
        assert torch.equal(o, ref)


def test_dit_batch_config_sampled_rows(M, oracle_mod):
    wl = W.dit_batch()
    out, lse = run_prefill(M, wl)
    rows = [0, 13, 31]
    ref, ref_lse = oracle(oracle_mod, wl, rows=rows)
    assert_close_to_oracle(out[rows], ref, torch.bfloat16, "dit rows")
    assert_lse_close(lse[rows], ref_lse, 2e-3)
    assert torch.isfinite(out).all()


CASES = [
    # B, Hq, Hkv, Lq, Lk, D
    (2, 4, 2, 300, 300, 128),
    (1, 2, 1, 129, 257, 64),
    (3, 8, 8, 70, 500, 128),
    (2, 6, 2, 256, 129, 64),
    (1, 4, 4, 1, 700, 128),
    (2, 16, 4, 384, 384, 128),
]


@pytest.mark.parametrize("mask", ["none", "bits", "kvlen", "segment", "bits+kvlen", "causal"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_random_cases_bf16(M, oracle_mod, mask, case):
    wl = W.random_case(sum(case) + len(mask), *case, dtype=torch.bfloat16, mask=mask)
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.bfloat16, f"{mask} {case}")
    assert_lse_close(lse, ref_lse, 2e-3)


@pytest.mark.parametrize("mask", ["none", "bits", "segment", "causal"])
@pytest.mark.parametrize("case", [(2, 8, 2, 300, 300, 128), (1, 2, 1, 129, 257, 64),
                                  (2, 4, 4, 200, 700, 128)], ids=lambda c: "x".join(map(str, c)))
def test_random_cases_fp16(M, oracle_mod, mask, case):
    wl = W.random_case(sum(case) + 3 * len(mask), *case, dtype=torch.float16, mask=mask)
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.float16, f"fp16 {mask} {case}")
    assert_lse_close(lse, ref_lse, 2e-3)


def test_causal_lq_shorter_than_lk(M, oracle_mod):
    """Causal queries as the last Lq of the Lk positions (a prefill chunk after a cache)."""
    wl = W.random_case(44, 2, 4, 2, 200, 640, 128, dtype=torch.bfloat16, mask="causal")
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.bfloat16, "causal chunk")
    assert_lse_close(lse, ref_lse, 2e-3)


@pytest.mark.parametrize("mask", ["bits", "segment", "causal"])
@pytest.mark.parametrize("case", [(2, 4, 2, 150, 200, 64), (1, 2, 2, 64, 1000, 128)],
                         ids=lambda c: "x".join(map(str, c)))
def test_random_cases_fp32(M, oracle_mod, mask, case):
    wl = W.random_case(sum(case), *case, dtype=torch.float32, mask=mask)
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.float32, f"fp32 {mask} {case}")
    assert_lse_close(lse, ref_lse, 1e-5)


@pytest.mark.parametrize("mask", ["none", "kvlen", "bits+kvlen"])
@pytest.mark.parametrize("case", [(1, 2, 1, 33, 37, 64), (2, 2, 2, 64, 64, 128), (1, 4, 2, 1, 65, 64),
                                  (2, 2, 1, 97, 191, 128)], ids=lambda c: "x".join(map(str, c)))
def test_fp32_key_tile_edges(M, oracle_mod, mask, case):
    """The fp32 kernel's double-buffered 64-key tiles at their edges: one
    partial tile, exactly one full tile, one full tile and one key, a ragged
    third tile; with key lengths that empty whole tiles of some rows."""
    wl = W.random_case(sum(case) + 7, *case, dtype=torch.float32, mask=mask)
    out, lse = run_prefill(M, wl)
    ref, ref_lse = oracle(oracle_mod, wl)
    assert_close_to_oracle(out, ref, torch.float32, f"fp32 {mask} {case}")
    assert_lse_close(lse, ref_lse, 1e-5)


def test_gqa_equals_repeated_heads(M):
    wl = W.random_case(5, 2, 8, 2, 200, 333, 128, dtype=torch.bfloat16, mask="bits")
    o1, l1 = run_prefill(M, wl)
    rep = W.Workload("rep", wl.q, wl.k.repeat_interleave(4, 1).contiguous(),
                     wl.v.repeat_interleave(4, 1).contiguous(), wl.scale, mask_bits=wl.mask_bits)
    o2, l2 = run_prefill(M, rep)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fully_masked_rows_give_zero(M):
    wl = W.random_case(9, 2, 4, 2, 200, 300, 128, dtype=torch.bfloat16, mask="kvlen")
    wl.kv_len[:] = torch.tensor([0, 5], dtype=torch.int32)
    out, lse = run_prefill(M, wl)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.isfinite(out[1]).all()


def test_strided_views(M, oracle_mod):
    """q/k/v/out as head-interleaved views ([B, L, H, D] storage)."""
    B, Hq, Hkv, L, D = 2, 4, 2, 200, 128
    g = torch.Generator().manual_seed(1)
    qs = torch.randn((B, L, Hq, D), generator=g).to(torch.bfloat16)
    ks = torch.randn((B, L, Hkv, D), generator=g).to(torch.bfloat16)
    vs = torch.randn((B, L, Hkv, D), generator=g).to(torch.bfloat16)
    qd, kd, vd = (t.cuda().transpose(1, 2) for t in (qs, ks, vs))
    outd = torch.empty((B, L, Hq, D), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    M.masked_gqa_attn_prefill(qd, kd, vd, outd, scale=0.1)
    torch.cuda.synchronize()
    ref, _, _ = oracle_mod.attention(qs.transpose(1, 2), ks.transpose(1, 2), vs.transpose(1, 2),
                                     scale=0.1)
    assert_close_to_oracle(outd, ref, torch.bfloat16, "strided")
