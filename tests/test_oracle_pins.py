"""Pins for the fp64 oracle: checks against facts fixed by the pages and by
mathematics, independent of the oracle's own code.

* hand-worked closed-form cases (tests/golden/hand_worked.json);
* library special case: torch's scaled_dot_product_attention in fp64 with
  enable_gqa and a boolean mask (rows with at least one allowed key);
* closed forms: one allowed key, scale 0, identical keys, a dominant score;
* invariants the pages state: masked slots add exact zeros (VoxCPM page,
  "Upstream-identical practice", attention bullet), packed block-diagonal
  rows equal each block run alone (OmniVoice page, "Memory & speed",
  packed_guidance paragraph), grouped KV heads equal explicitly repeated
  heads (OmniVoice page, "Upstream-identical practice", attention-mask
  bullet), truncating the key range past the last allowed key changes nothing;
* brute force at 50 significant digits on tiny inputs (mpmath).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _arr(x):
    return np.array(x, dtype=np.float64)


def _run(oracle_mod, wl, **kw):
    out, lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks(), **kw)
    return out, lse


# --- hand-worked golden cases ----------------------------------------------

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_worked(oracle_mod, case):
    B, Lq, Lk = case["B"], case["Lq"], case["Lk"]
    masks = {}
    if "mask_bool" in case:
        masks["mask_bits"] = W.pack_bool_mask(torch.tensor(case["mask_bool"], dtype=torch.bool))
    if "kv_len" in case:
        masks["kv_len"] = torch.tensor(case["kv_len"], dtype=torch.int32)
    if "seg" in case:
        masks["seg_q"] = torch.tensor(case["seg"], dtype=torch.int32)
        masks["seg_k"] = torch.tensor(case["seg"], dtype=torch.int32)
    out, lse, _ = oracle_mod.attention(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                                       scale=case["scale"], **masks)
    exp_out = _arr(case["out"])
    exp_lse = np.array([[[float(x) for x in r] for r in h] for h in case["lse"]])
    np.testing.assert_allclose(out, exp_out, rtol=1e-14, atol=1e-14)
    fin = np.isfinite(exp_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], exp_lse[fin], rtol=1e-14, atol=1e-14)
    assert np.all(lse[~fin] == -np.inf)


# --- library special case: torch SDPA in fp64 ------------------------------

@pytest.mark.parametrize("mask", ["none", "bits", "kvlen", "segment", "bits+kvlen"])
@pytest.mark.parametrize("shape", [(2, 4, 2, 33, 70, 16), (2, 6, 3, 17, 17, 8), (3, 2, 1, 5, 129, 32)])
def test_matches_torch_sdpa_fp64(oracle_mod, mask, shape):
    B, Hq, Hkv, Lq, Lk, D = shape
    wl = W.random_case(11 + Lq + Lk, B, Hq, Hkv, Lq, Lk, D, torch.float64, mask=mask)
    out, lse = _run(oracle_mod, wl)
    allowed = wl.allowed()  # [B, Lq, Lk]
    ref = torch.nn.functional.scaled_dot_product_attention(
        wl.q, wl.k, wl.v, attn_mask=allowed[:, None], scale=wl.scale, enable_gqa=True)
    rows = allowed.any(-1)  # [B, Lq]
    sel = rows[:, None, :].expand(B, Hq, Lq).numpy()
    np.testing.assert_allclose(out[sel], ref.numpy()[sel], rtol=1e-12, atol=1e-12)
    # LSE: logsumexp of the masked scores, via torch
    kk = wl.k.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("bhid,bhjd->bhij", wl.q, kk) * wl.scale
    s = s.masked_fill(~allowed[:, None], -math.inf)
    ref_lse = torch.logsumexp(s, dim=-1).numpy()
    np.testing.assert_allclose(lse[sel], ref_lse[sel], rtol=1e-12, atol=1e-12)
    assert np.all(out[~sel] == 0.0) and np.all(lse[~sel] == -np.inf)


# --- closed forms ----------------------------------------------------------

def test_single_allowed_key_returns_its_value_exactly(oracle_mod):
    B, Hq, Hkv, L, D = 2, 4, 2, 40, 16
    g, q, k, v = W.random_qkv(5, B, Hq, Hkv, L, L, D, torch.float64)
    j = torch.randint(0, L, (B, L), generator=g)
    mask = torch.zeros((B, L, L), dtype=torch.bool)
    mask.scatter_(2, j[..., None], True)
    out, lse, _ = oracle_mod.attention(q, k, v, scale=0.3, mask_bits=W.pack_bool_mask(mask))
    for b in range(B):
        for h in range(Hq):
            gk = h // (Hq // Hkv)
            for i in range(L):
                jj = int(j[b, i])
                assert np.array_equal(out[b, h, i], v[b, gk, jj].numpy())
                s = 0.3 * float((q[b, h, i] * k[b, gk, jj]).sum())
                assert lse[b, h, i] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_zero_scale_gives_mean_of_allowed_values(oracle_mod):
    wl = W.random_case(21, 2, 4, 2, 24, 50, 8, torch.float64, mask="bits")
    out, lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=0.0, mask_bits=wl.mask_bits)
    a = wl.allowed()
    for b in range(2):
        for h in range(4):
            for i in range(24):
                idx = torch.nonzero(a[b, i]).flatten()
                if len(idx) == 0:
                    assert np.all(out[b, h, i] == 0) and lse[b, h, i] == -np.inf
                    continue
                mean = wl.v[b, h // 2, idx].mean(0).numpy()
                np.testing.assert_allclose(out[b, h, i], mean, rtol=1e-13, atol=1e-13)
                assert lse[b, h, i] == pytest.approx(math.log(len(idx)), rel=1e-13)


def test_identical_keys_give_mean(oracle_mod):
    B, Hq, Hkv, L, D = 1, 2, 1, 9, 8
    g, q, k, v = W.random_qkv(3, B, Hq, Hkv, L, L, D, torch.float64)
    k[:] = k[:, :, :1, :]
    out, _, _ = oracle_mod.attention(q, k, v, scale=1.7)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0].mean(0).numpy(), rtol=1e-13, atol=1e-13)


def test_dominant_score_selects_its_value(oracle_mod):
    B, Hq, Hkv, L, D = 1, 1, 1, 6, 4
    q = torch.zeros((B, Hq, 1, D), dtype=torch.float64)
    q[..., 0] = 1.0
    k = torch.zeros((B, Hkv, L, D), dtype=torch.float64)
    k[0, 0, :, 0] = torch.tensor([0.0, 3.0, -2.0, 103.5, 1.0, 2.5])
    v = torch.arange(L * D, dtype=torch.float64).reshape(B, Hkv, L, D)
    out, lse, _ = oracle_mod.attention(q, k, v, scale=1.0)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 3].numpy(), rtol=1e-12)
    assert lse[0, 0, 0] == pytest.approx(103.5, abs=1e-12)


# --- invariants stated on the pages ----------------------------------------

def test_masked_slots_add_exact_zeros(oracle_mod):
    """Refilling masked K/V with arbitrary finite values leaves every bit."""
    wl = W.static_cache_decode(seed=77, B=3, capacity=512, lo=40, hi=300, dtype=torch.float64)
    out1, lse1 = _run(oracle_mod, wl)
    g = torch.Generator().manual_seed(9)
    k2, v2 = wl.k.clone(), wl.v.clone()
    for b, n in enumerate(wl.info["filled"]):
        k2[b, :, n:] = torch.randn(k2[b, :, n:].shape, generator=g) * 1e3
        v2[b, :, n:] = -torch.randn(v2[b, :, n:].shape, generator=g) * 1e4
    out2, lse2, _ = oracle_mod.attention(wl.q, k2, v2, scale=wl.scale, kv_len=wl.kv_len)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_packed_rows_equal_blocks_alone(oracle_mod):
    B, Hq, Hkv, D = 1, 4, 2, 16
    L1, L2 = 37, 21
    g, q, k, v = W.random_qkv(31, B, Hq, Hkv, L1 + L2, L1 + L2, D, torch.float64)
    seg = torch.zeros((1, L1 + L2), dtype=torch.int32)
    seg[:, L1:] = 1
    out, lse, _ = oracle_mod.attention(q, k, v, scale=0.25, seg_q=seg, seg_k=seg)
    for lo, hi in ((0, L1), (L1, L1 + L2)):
        o1, l1, _ = oracle_mod.attention(q[:, :, lo:hi], k[:, :, lo:hi], v[:, :, lo:hi], scale=0.25)
        assert np.array_equal(out[:, :, lo:hi], o1)
        assert np.array_equal(lse[:, :, lo:hi], l1)


def test_gqa_equals_repeated_kv_heads(oracle_mod):
    wl = W.random_case(41, 2, 6, 2, 19, 45, 8, torch.float64, mask="bits")
    out, lse = _run(oracle_mod, wl)
    kr = wl.k.repeat_interleave(3, dim=1)
    vr = wl.v.repeat_interleave(3, dim=1)
    out2, lse2, _ = oracle_mod.attention(wl.q, kr, vr, scale=wl.scale, mask_bits=wl.mask_bits)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_truncation_past_last_allowed_key(oracle_mod):
    wl = W.static_cache_decode(seed=5, B=4, Hq=4, Hkv=2, D=16, capacity=300, lo=20, hi=180,
                               dtype=torch.float64)
    out, lse = _run(oracle_mod, wl)
    last = max(wl.info["filled"])
    for Lk in (last, last + 1, last + 63, 299):
        o2, l2, _ = oracle_mod.attention(wl.q, wl.k[:, :, :Lk], wl.v[:, :, :Lk], scale=wl.scale,
                                         kv_len=wl.kv_len)
        assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_fully_masked_rows_are_zero(oracle_mod):
    wl = W.random_case(8, 2, 2, 1, 5, 7, 4, torch.float64, mask="kvlen")
    wl.kv_len[:] = 0
    out, lse = _run(oracle_mod, wl)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_brute_force_high_precision(oracle_mod):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    wl = W.random_case(61, 1, 2, 1, 3, 6, 3, torch.float64, mask="bits", density=0.6)
    out, lse = _run(oracle_mod, wl)
    a = wl.allowed()
    for h in range(2):
        for i in range(3):
            keys = [j for j in range(6) if a[0, i, j]]
            if not keys:
                assert lse[0, h, i] == -np.inf
                continue
            s = [mpmath.mpf(wl.scale) * mpmath.fsum(mpmath.mpf(float(wl.q[0, h, i, d])) *
                                                    mpmath.mpf(float(wl.k[0, 0, j, d])) for d in range(3))
                 for j in keys]
            den = mpmath.fsum(mpmath.e ** x for x in s)
            for d in range(3):
                num = mpmath.fsum(mpmath.e ** x * mpmath.mpf(float(wl.v[0, 0, j, d]))
                                  for x, j in zip(s, keys))
                assert float(num / den) == pytest.approx(out[0, h, i, d], rel=1e-13, abs=1e-13)
            assert float(mpmath.log(den)) == pytest.approx(lse[0, h, i], rel=1e-13, abs=1e-13)


# --- workload shapes match the stated configurations -------------------------

def test_workload_algorithmic_counts():
    wl = W.padded_cfg()
    assert wl.flops() == pytest.approx(11.81e9, rel=1e-3)
    assert wl.nonempty_tile_flops() == wl.flops()
    wk = W.padded_cfg(variant="kvlen")
    assert torch.equal(wk.allowed(), wl.allowed())
    wp = W.packed_guidance()
    assert wp.flops() == pytest.approx(9.80e9, rel=1e-3)
    wt = W.tiny_fp32()
    assert int(wt.allowed()[1].sum()) == 128 * 48 and bool(wt.allowed()[1, :, 80:].all())


def test_pack_unpack_roundtrip():
    g = torch.Generator().manual_seed(1)
    m = torch.rand((3, 5, 77), generator=g) < 0.5
    words = W.pack_bool_mask(m)
    assert words.shape == (3, 5, 3) and words.dtype == torch.int32
    assert torch.equal(W.unpack_bits(words, 77), m)
    # bit order: key 0 is the least significant bit of word 0
    one = torch.zeros((1, 1, 40), dtype=torch.bool)
    one[0, 0, 0] = True
    one[0, 0, 33] = True
    w = W.pack_bool_mask(one)
    assert int(w[0, 0, 0]) == 1 and int(w[0, 0, 1]) == 2


# --- causal form (VoxCPM page, "Upstream-identical practice": causal prefill)

@pytest.mark.parametrize("shape", [(2, 4, 2, 33, 33, 16), (1, 6, 3, 70, 70, 8)])
@pytest.mark.parametrize("mask", ["none", "bits"])
def test_causal_matches_torch_sdpa_fp64(oracle_mod, shape, mask):
    B, Hq, Hkv, Lq, Lk, D = shape
    wl = W.random_case(7 + Lq, B, Hq, Hkv, Lq, Lk, D, torch.float64, mask=mask)
    out, lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, causal=True,
                                       mask_bits=wl.mask_bits)
    tril = torch.ones((Lq, Lk), dtype=torch.bool).tril()
    allowed = tril[None].expand(B, Lq, Lk).clone()
    if wl.mask_bits is not None:
        allowed &= W.unpack_bits(wl.mask_bits, Lk)
    if mask == "none":  # library causal flag itself
        ref = torch.nn.functional.scaled_dot_product_attention(
            wl.q, wl.k, wl.v, is_causal=True, scale=wl.scale, enable_gqa=True)
    else:
        ref = torch.nn.functional.scaled_dot_product_attention(
            wl.q, wl.k, wl.v, attn_mask=allowed[:, None], scale=wl.scale, enable_gqa=True)
    sel = allowed.any(-1)[:, None, :].expand(B, Hq, Lq).numpy()
    np.testing.assert_allclose(out[sel], ref.numpy()[sel], rtol=1e-12, atol=1e-12)


def test_causal_first_row_and_single_query(oracle_mod):
    g, q, k, v = W.random_qkv(2, 1, 2, 1, 9, 9, 4, torch.float64)
    out, lse, _ = oracle_mod.attention(q, k, v, scale=0.7, causal=True)
    # row 0 sees key 0 only: its value, exactly
    assert np.array_equal(out[0, 0, 0], v[0, 0, 0].numpy())
    assert np.array_equal(out[0, 1, 0], v[0, 0, 0].numpy())
    # one query over a 9-slot cache is the last position: every key allowed
    o1, l1, _ = oracle_mod.attention(q[:, :, -1:], k, v, scale=0.7, causal=True)
    o2, l2, _ = oracle_mod.attention(q[:, :, -1:], k, v, scale=0.7)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---- rotary position embedding (F5-TTS page: interleaved pairs on the first
# pe_attn_head heads; OmniVoice page, "Parity results", and VoxCPM page,
# precision bullet: fp32 inverse frequencies;
# OmniVoice page, packed_guidance: positions restart per packed sequence) ----

def _rope_inputs(seed, B=2, H=3, L=5, D=8):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, L, D, generator=g, dtype=torch.float64).numpy()


def test_rope_hand_worked_pairs(oracle_mod):
    # interleaved: (x0, x1) rotates by pos * f0, (x2, x3) by pos * f1
    x = np.array([[[[1.0, 0.0, 0.0, 1.0]]]])
    f = np.array([1.0, 0.5], np.float32)
    y = oracle_mod.rope(x, inv_freq=f, positions=np.array([[1]], np.int32), interleaved=True)
    assert np.allclose(y[0, 0, 0], [math.cos(1), math.sin(1), -math.sin(0.5), math.cos(0.5)],
                       rtol=0, atol=1e-15)
    # half-split: (x0, x2) rotates by f0, (x1, x3) by f1
    y = oracle_mod.rope(x, inv_freq=f, positions=np.array([[1]], np.int32), interleaved=False)
    assert np.allclose(y[0, 0, 0], [math.cos(1), -math.sin(0.5), math.sin(1), math.cos(0.5)],
                       rtol=0, atol=1e-15)


def test_rope_position_zero_is_identity(oracle_mod):
    x = _rope_inputs(1)
    f = (10000.0 ** (-np.arange(0, 8, 2) / 8)).astype(np.float32)
    y = oracle_mod.rope(x, inv_freq=f, positions=np.zeros((2, 5), np.int32))
    assert np.array_equal(y, x)


def test_rope_quarter_turn(oracle_mod):
    # angle fl32(pi/2): (a, c) -> (-c, a) up to the 4.4e-8 rounding of pi/2
    x = _rope_inputs(2, D=2)
    y = oracle_mod.rope(x, inv_freq=np.array([np.float32(math.pi / 2)]),
                        positions=np.ones((2, 5), np.int32), interleaved=True)
    assert np.allclose(y[..., 0], -x[..., 1], atol=1e-7) and np.allclose(y[..., 1], x[..., 0], atol=1e-7)


@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_keeps_pair_norms(oracle_mod, interleaved):
    x = _rope_inputs(3)
    f = (10000.0 ** (-np.arange(0, 8, 2) / 8)).astype(np.float32)
    pos = np.array([[0, 7, 100, 4095, 8191], [3, 1, 2, 5, 9]], np.int32)
    y = oracle_mod.rope(x, inv_freq=f, positions=pos, interleaved=interleaved)
    if interleaved:
        n0, n1 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2, y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    else:
        n0, n1 = x[..., :4] ** 2 + x[..., 4:] ** 2, y[..., :4] ** 2 + y[..., 4:] ** 2
    assert np.allclose(n1, n0, rtol=1e-13, atol=0)
    assert not np.allclose(y, x)


def test_rope_layouts_are_one_permutation(oracle_mod):
    # interleaved pairs (2i, 2i+1) are half-split pairs (i, i + r/2) of the
    # feature-permuted vector
    x = _rope_inputs(4)
    f = np.array([0.9, 0.3, 0.05, 0.001], np.float32)
    pos = np.array([[0, 1, 2, 30, 500], [5, 4, 3, 2, 1]], np.int32)
    perm = np.array([0, 2, 4, 6, 1, 3, 5, 7])  # interleaved index of half-split slot
    yi = oracle_mod.rope(x, inv_freq=f, positions=pos, interleaved=True)
    yh = oracle_mod.rope(np.ascontiguousarray(x[..., perm]), inv_freq=f, positions=pos,
                         interleaved=False)
    assert np.array_equal(yi[..., perm], yh)


def test_rope_partial_dims_and_heads(oracle_mod):
    x = _rope_inputs(5, H=4, D=8)
    f = np.array([0.5, 0.25], np.float32)
    y = oracle_mod.rope(x, inv_freq=f, rot_dim=4, heads=1, interleaved=True)
    assert np.array_equal(y[:, 1:], x[:, 1:])           # heads past `heads` untouched
    assert np.array_equal(y[:, :1, :, 4:], x[:, :1, :, 4:])  # features past rot_dim untouched
    assert not np.array_equal(y[:, :1, 1:, :4], x[:, :1, 1:, :4])
    # positions default to the row index
    pos = np.tile(np.arange(5, dtype=np.int32), (2, 1))
    y2 = oracle_mod.rope(x, inv_freq=f, rot_dim=4, heads=1, interleaved=True, positions=pos)
    assert np.array_equal(y, y2)


def test_rope_angles_add_and_scores_see_only_offsets(oracle_mod):
    # power-of-two frequencies make every fp32 angle exact, so rotations
    # compose (R(p) R(q) = R(p + q)) and q.k after rotation depends only on
    # the position difference
    x = _rope_inputs(6, B=1, H=1, L=1, D=8)
    k = _rope_inputs(7, B=1, H=1, L=1, D=8)
    f = np.array([1.0, 0.5, 0.125, 2 ** -10], np.float32)

    def rot(v, p):
        return oracle_mod.rope(v, inv_freq=f, positions=np.array([[p]], np.int32), interleaved=False)
    assert np.allclose(rot(rot(x, 37), 1000), rot(x, 1037), rtol=0, atol=1e-12)
    s1 = float((rot(x, 50) * rot(k, 20)).sum())
    s2 = float((rot(x, 1050) * rot(k, 1020)).sum())
    assert abs(s1 - s2) < 1e-12 and abs(s1 - float((x * k).sum())) > 1e-3


def test_rope_angle_is_the_fp32_product(oracle_mod):
    # theta = fl32(pos * f): with f = fl32(0.1) and pos = 3 the product rounds
    # to a different float than 3 * 0.1 in fp64
    f = np.float32(0.1)
    theta32 = float(np.float32(np.float32(3) * f))
    assert theta32 != 3 * float(f)
    x = np.array([[[[1.0, 0.0]]]])
    y = oracle_mod.rope(x, inv_freq=np.array([f]), positions=np.array([[3]], np.int32))
    assert y[0, 0, 0, 0] == math.cos(theta32) and y[0, 0, 0, 1] == math.sin(theta32)



# ---- RMS normalisation of q and k (OmniVoice page, "Parity results": the shared
# Qwen decoder normalises q and k separately before the rotation) ----

def test_rms_norm_hand_worked(oracle_mod):
    # x = (3, 4): mean of squares 12.5, so y = x / sqrt(12.5) * w
    x = np.array([[[[3.0, 4.0]]]])
    y = oracle_mod.rms_norm(x, weight=np.array([1.0, 2.0], np.float32), eps=0.0)
    s = math.sqrt(12.5)
    assert np.allclose(y[0, 0, 0], [3.0 / s, 8.0 / s], rtol=0, atol=1e-15)
    # eps enters under the root: x = (1, 1), eps = 3 -> 1 / sqrt(1 + 3) = 1/2
    y = oracle_mod.rms_norm(np.ones((1, 1, 1, 2)), weight=np.ones(2, np.float32), eps=3.0)
    assert np.array_equal(y, np.full((1, 1, 1, 2), 0.5))


def test_rms_norm_unit_mean_square_and_scale_invariance(oracle_mod):
    x = _rope_inputs(8, H=3, D=16)
    y = oracle_mod.rms_norm(x, weight=np.ones(16, np.float32), eps=0.0)
    assert np.allclose((y ** 2).mean(-1), 1.0, rtol=1e-14, atol=0)
    y2 = oracle_mod.rms_norm(7.5 * x, weight=np.ones(16, np.float32), eps=0.0)
    assert np.allclose(y2, y, rtol=1e-13, atol=1e-15)


def test_rms_norm_matches_library_and_spares_heads(oracle_mod):
    x = _rope_inputs(9, B=2, H=4, L=5, D=8)
    w = np.linspace(0.5, 2.0, 8).astype(np.float32)
    y = oracle_mod.rms_norm(x, weight=w, eps=1e-6, heads=2)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x[:, :2]), (8,),
                                       weight=torch.from_numpy(w).double(), eps=1e-6)
    assert np.allclose(y[:, :2], ref.numpy(), rtol=1e-14, atol=1e-15)
    assert np.array_equal(y[:, 2:], x[:, 2:])  # heads past `heads` untouched


def test_rms_norm_then_rope_keeps_the_normalised_length(oracle_mod):
    # the rotation after the norm preserves each vector's length, so with a
    # unit weight every rotated head vector has mean square 1
    x = _rope_inputs(10, H=2, D=8)
    f = (10000.0 ** (-np.arange(0, 8, 2) / 8)).astype(np.float32)
    pos = np.array([[0, 9, 99, 999, 4095], [1, 2, 3, 4, 5]], np.int32)
    y = oracle_mod.rope(oracle_mod.rms_norm(x, weight=np.ones(8, np.float32), eps=0.0),
                        inv_freq=f, positions=pos, interleaved=False)
    assert np.allclose((y ** 2).mean(-1), 1.0, rtol=1e-13, atol=0)
