"""The rotary embedding (and the Qwen3-style RMS normalisation of q and k)
fused into the attention kernels.

Pages: F5-TTS page, module table and "Upstream-identical practice"
(interleaved pairs, only the first pe_attn_head heads rotate); OmniVoice
page, "Parity results" (fp32 inverse frequencies; q and k normalised
separately before the rotation); VoxCPM page, "Memory & speed" (each decode
step advances one position against the static cache).

* A fused call gives the same bits as the standalone masked_gqa_rope on q
  (and on the new key row) followed by the plain attention call.
* It matches the fp64 oracle composed from its pinned pieces:
  rms_norm -> rope -> attention.
"""
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


def inv_freq_table(rot_dim, base=10000.0):
    return (base ** (-torch.arange(0, rot_dim, 2, dtype=torch.float64) / rot_dim)).to(torch.float32)


def norm_weight(seed, D):
    g = torch.Generator().manual_seed(seed)
    return (0.5 + torch.rand(D, generator=g)).to(torch.float32)


def oracle_qk(oracle_mod, x, f, pos, rot, heads, inter, w, eps):
    """The oracle's normalised and rotated copy of x (fp64)."""
    y = x if w is None else oracle_mod.rms_norm(x, weight=w, eps=eps, heads=heads)
    return oracle_mod.rope(y, inv_freq=f, positions=pos, rot_dim=rot, heads=heads, interleaved=inter)


PREFILL = [
    # (B, Hq, Hkv, L, D, mask, rot_dim, q_heads, interleaved, norm)
    (2, 16, 8, 1024, 128, "bits", 128, 16, False, True),    # OmniVoice-shaped padded CFG, Qwen3 norm
    (2, 16, 4, 700, 128, "segment", 128, 16, False, False),  # DiT-shaped segments, ragged length
    (1, 8, 8, 300, 64, "none", 64, 1, True, False),          # F5: one rotated head, interleaved
    (2, 4, 2, 257, 128, "causal", 64, 4, False, True),       # partial rotary dim (half-split)
    (1, 4, 2, 200, 64, "kvlen", 32, 2, True, True),          # partial, interleaved, 2 of 4 heads
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "-".join(map(str, c)))
def test_prefill_fused_rope_equals_standalone_then_attention(M, oracle_mod, dtype, case):
    B, Hq, Hkv, L, D, mask, rot, qh, inter, norm = case
    wl = W.random_case(B + L + rot, B, Hq, Hkv, L, L, D, dtype=dtype, mask=mask)
    f = inv_freq_table(rot)
    g = torch.Generator().manual_seed(L)
    pos = torch.randint(0, 4096, (B, L), generator=g, dtype=torch.int32)
    wq = norm_weight(1, D) if norm else None
    wk = norm_weight(2, D) if norm else None
    eps = 1e-6
    d = to_device(wl)
    fd, pd = f.cuda(), pos.cuda()
    wqd = wq.cuda() if norm else None
    wkd = wk.cuda() if norm else None
    # keys rotated (and normalised) once by the standalone kernel
    k_rot = d["k"].clone()
    M.masked_gqa_rope(k_rot, fd, positions=pd, rot_dim=rot, heads=Hkv if qh == Hq else max(1, qh * Hkv // Hq),
                      interleaved=inter, norm_weight=wkd, norm_eps=eps)
    masks = dict(mask_bits=d["mask_bits"], kv_len=d["kv_len"], seg_q=d["seg_q"], seg_k=d["seg_k"],
                 causal=wl.causal)
    # unfused: standalone rotation of q, plain prefill
    q_rot = d["q"].clone()
    M.masked_gqa_rope(q_rot, fd, positions=pd, rot_dim=rot, heads=qh, interleaved=inter,
                      norm_weight=wqd, norm_eps=eps)
    lse1 = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
    o1 = M.masked_gqa_attn_prefill(q_rot, k_rot, d["v"], scale=wl.scale, lse=lse1, **masks)
    # fused
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse2 = torch.empty_like(lse1)
    o2 = M.masked_gqa_attn_prefill_rope(d["q"], k_rot, d["v"], inv_freq=fd, positions=pd, rot_dim=rot,
                                        interleaved=inter, q_heads=qh, q_norm_weight=wqd, norm_eps=eps,
                                        scale=wl.scale, lse=lse2, dev_error=err, **masks)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    # against the oracle, from the original inputs
    kh = Hkv if qh == Hq else max(1, qh * Hkv // Hq)
    q64 = oracle_qk(oracle_mod, wl.q, f, pos, rot, qh, inter, wq, eps)
    k64 = oracle_qk(oracle_mod, wl.k, f, pos, rot, kh, inter, wk, eps)
    ref, ref_lse, _ = oracle_mod.attention(q64, k64, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(o2, ref, dtype, f"fused prefill {case}")
    # the GPU rounds the transformed q and k to the I/O type (the oracle keeps
    # them exact): a score moves by up to scale * |q| |k| * 2^-8 (about 0.04
    # for normalised 128-wide heads), and the LSE with it
    assert_lse_close(lse2, ref_lse, 2e-2)


DECODE_ROPE = [  # Hq, Hkv, D, rot_dim
    (16, 2, 64, 64),    # the static-cache decode heads: 8 query rows + the key row per CTA
    (8, 2, 128, 64),    # partial rotary dim, 4 query rows per CTA
    (4, 4, 128, 128),   # one query row per CTA
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("norm", ["none", "both", "q", "k"])
@pytest.mark.parametrize("inter", [False, True])
@pytest.mark.parametrize("shape", DECODE_ROPE, ids=lambda c: "x".join(map(str, c)))
def test_decode_step_fused_rope_equals_standalone_then_append(M, oracle_mod, dtype, norm, inter, shape):
    Hq, Hkv, D, rot = shape
    wl = W.static_cache_decode(seed=71 + D + Hq, variant="span", B=4, Hq=Hq, Hkv=Hkv, D=D,
                               capacity=3000, lo=100, hi=2900, dtype=dtype)
    B = wl.shape[0]
    f = inv_freq_table(rot)
    wq = norm_weight(3, D) if norm in ("both", "q") else None
    wk = norm_weight(4, D) if norm in ("both", "k") else None
    g = torch.Generator().manual_seed(9)
    kn = torch.randn((B, Hkv, 1, D), generator=g).to(dtype)
    vn = torch.randn((B, Hkv, 1, D), generator=g).to(dtype)
    q, k, v, kvl = (t.cuda() for t in (wl.q, wl.k, wl.v, wl.kv_len))
    fd = f.cuda()
    wqd = wq.cuda() if wq is not None else None
    wkd = wk.cuda() if wk is not None else None
    pos = kvl.clone()  # the new token's position: its cache slot
    # unfused: rotate q and the new key row (positions [B, 1] = the slot), then append
    q_rot, kn_rot = q.clone(), kn.cuda().clone()
    M.masked_gqa_rope(q_rot, fd, positions=pos[:, None].contiguous(), rot_dim=rot, norm_weight=wqd,
                      interleaved=inter)
    M.masked_gqa_rope(kn_rot, fd, positions=pos[:, None].contiguous(), rot_dim=rot, norm_weight=wkd,
                      interleaved=inter)
    k1, v1 = k.clone(), v.clone()
    len1 = torch.zeros_like(kvl)
    o1 = M.masked_gqa_attn_decode_append(q_rot, k1, v1, kn_rot, vn.cuda(), kvl, kv_len_out=len1,
                                         scale=wl.scale)
    # fused
    k2, v2 = k.clone(), v.clone()
    len2 = torch.zeros_like(kvl)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2 = M.masked_gqa_attn_decode_append_rope(q, k2, v2, kn.cuda(), vn.cuda(), kvl, inv_freq=fd,
                                              rot_dim=rot, interleaved=inter, q_norm_weight=wqd,
                                              k_norm_weight=wkd, kv_len_out=len2, scale=wl.scale,
                                              dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(len1, len2)
    # against the oracle: the cache after the append holds the rotated new row
    pos_c = wl.kv_len.clone()
    q64 = oracle_qk(oracle_mod, wl.q, f, pos_c[:, None], rot, Hq, inter, wq, 1e-6)
    kn64 = oracle_qk(oracle_mod, kn, f, pos_c[:, None], rot, Hkv, inter, wk, 1e-6)
    kc = wl.k.double().numpy().copy()
    vc = wl.v.double().numpy().copy()
    for b in range(B):
        n = int(wl.kv_len[b])
        kc[b, :, n] = kn64[b, :, 0]
        vc[b, :, n] = vn[b, :, 0].double().numpy()
    ref, _, _ = oracle_mod.attention(q64, kc, vc, scale=wl.scale, kv_len=wl.kv_len + 1)
    assert_close_to_oracle(o2, ref, dtype, "fused decode step")


def test_decode_steps_ping_pong_with_fused_rope(M, oracle_mod):
    """Three fused steps in a row: each new token at its own slot position."""
    wl = W.static_cache_decode(seed=72, variant="span", B=2, Hq=16, Hkv=2, D=128, capacity=800,
                               lo=10, hi=500)
    B, Hq, Hkv, _, Lk, D = wl.shape
    f = inv_freq_table(D)
    q, k, v = (t.cuda() for t in (wl.q, wl.k, wl.v))
    lens = [wl.kv_len.cuda(), torch.zeros_like(wl.kv_len).cuda()]
    ws = M.new_decode_workspace(q, k, v, kv_len=lens[0])
    kc, vc = wl.k.double().numpy().copy(), wl.v.double().numpy().copy()
    for step in range(3):
        g = torch.Generator().manual_seed(200 + step)
        kn = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16)
        cur, nxt = lens[step % 2], lens[(step + 1) % 2]
        n_before = cur.cpu().clone()
        out = M.masked_gqa_attn_decode_append_rope(q, k, v, kn.cuda(), vn.cuda(), cur, workspace=ws,
                                                   inv_freq=f.cuda(), kv_len_out=nxt, scale=wl.scale)
        torch.cuda.synchronize()
        kn64 = oracle_mod.rope(kn, inv_freq=f, positions=n_before[:, None])
        for b in range(B):
            kc[b, :, int(n_before[b])] = kn64[b, :, 0]
            vc[b, :, int(n_before[b])] = vn[b, :, 0].double().numpy()
        q64 = oracle_mod.rope(wl.q, inv_freq=f, positions=n_before[:, None])
        ref, _, _ = oracle_mod.attention(q64, kc, vc, scale=wl.scale, kv_len=n_before + 1)
        assert_close_to_oracle(out, ref, torch.bfloat16, f"step {step}")
        assert torch.equal(nxt.cpu(), n_before + 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("case", [(2, 16, 300, 128, 128, 16, False), (1, 4, 77, 64, 32, 2, True),
                                  (2, 8, 64, 128, 64, 8, False)], ids=lambda c: "x".join(map(str, c)))
def test_standalone_rope_with_norm_matches_oracle(M, oracle_mod, dtype, case):
    B, H, L, D, rot, heads, inter = case
    g = torch.Generator().manual_seed(L + D)
    x = torch.randn(B, H, L, D, generator=g).to(dtype)
    f = inv_freq_table(rot)
    w = norm_weight(5, D)
    pos = torch.randint(0, 8192, (B, L), generator=g, dtype=torch.int32)
    xd = x.cuda()
    M.masked_gqa_rope(xd, f.cuda(), positions=pos.cuda(), rot_dim=rot, heads=heads, interleaved=inter,
                      norm_weight=w.cuda(), norm_eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle_qk(oracle_mod, x, f, pos, rot, heads, inter, w, 1e-5)
    got = xd.cpu()
    if dtype == torch.float32:
        assert_close_to_oracle(xd, ref, dtype, f"rope+norm {case}")
    else:
        u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11
        err = np.abs(got.double().numpy() - ref)
        assert np.all(err <= u * np.abs(ref) + 2e-5), float((err - u * np.abs(ref)).max())
    assert torch.equal(got[:, heads:], x[:, heads:])
