"""Parity of the rotary-position-embedding kernel against the fp64 oracle, and
the properties the pages fix: only the first `heads` heads and `rot_dim`
features rotate (F5-TTS page, pe_attn_head), and under packing each
sequence's positions restart at 0 (OmniVoice page, packed_guidance), so a
packed row rotates exactly like its sequences alone."""
import numpy as np
import pytest
import torch

from _util import assert_close_to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import masked_gqa_attention_gb300 as M
    M.build_library()
    return M


def inv_freq_table(rot_dim, base=10000.0):
    # the usual table, built in fp32 (OmniVoice page, "Parity results": it stays fp32)
    return (base ** (-torch.arange(0, rot_dim, 2, dtype=torch.float64) / rot_dim)).to(torch.float32)


def make_x(seed, B, H, L, D, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, L, D, generator=g, dtype=torch.float32).to(dtype)


CASES = [  # B, H, L, D, rot_dim, heads
    (2, 16, 1024, 128, 128, 16),   # language-model q at the padded-CFG shape
    (2, 8, 1024, 128, 64, 8),      # partial rotary dim
    (1, 3, 77, 64, 32, 1),         # F5 DiT: one rotated head (pe_attn_head = 1)
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_rope_matches_oracle(M, oracle_mod, dtype, interleaved, case):
    B, H, L, D, rot, heads = case
    x = make_x(11 + L, B, H, L, D, dtype)
    f = inv_freq_table(rot)
    g = torch.Generator().manual_seed(5)
    pos = torch.randint(0, 8192, (B, L), generator=g, dtype=torch.int32)
    ref = oracle_mod.rope(x, inv_freq=f, positions=pos, rot_dim=rot, heads=heads,
                          interleaved=interleaved)
    xd = x.cuda()
    M.masked_gqa_rope(xd, f.cuda(), positions=pos.cuda(), rot_dim=rot, heads=heads,
                      interleaved=interleaved)
    torch.cuda.synchronize()
    assert_close_to_oracle(xd, ref, dtype, f"rope {case}")
    got = xd.cpu()
    if dtype != torch.float32:
        # per element: rounding the fp32 result to the output type (unit
        # roundoff 2^-8 for bf16, 2^-11 for fp16) plus the fp32 arithmetic: a
        # few ulp of |a| + |c|, and the sine and cosine's own error (at most
        # about 5e-7 after the reduction by 2 pi) times |a| + |c| <= 10 here
        u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11
        err = np.abs(got.double().numpy() - ref)
        assert np.all(err <= u * np.abs(ref) + 1e-5), float((err - u * np.abs(ref)).max())
    # what must not rotate is bit-for-bit the input
    assert torch.equal(got[:, heads:], x[:, heads:])
    assert torch.equal(got[..., rot:], x[..., rot:])


def test_rope_default_positions_are_row_index(M):
    x = make_x(3, 2, 4, 300, 64, torch.bfloat16).cuda()
    f = inv_freq_table(64).cuda()
    a = M.masked_gqa_rope(x.clone(), f)
    pos = torch.arange(300, dtype=torch.int32, device="cuda").repeat(2, 1).contiguous()
    b = M.masked_gqa_rope(x.clone(), f, positions=pos)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_rope_packed_row_equals_sequences_alone(M):
    # cond (1024) and uncond target (384) packed in one row, positions 0.. per sequence
    B, H, D = 1, 8, 128
    xc, xu = make_x(21, B, H, 1024, D, torch.bfloat16).cuda(), make_x(22, B, H, 384, D, torch.bfloat16).cuda()
    f = inv_freq_table(D).cuda()
    packed, _ = M.masked_gqa_pack_pair(xc, xu)
    pos = torch.cat([torch.arange(1024), torch.arange(384)]).to(torch.int32)[None].cuda().contiguous()
    M.masked_gqa_rope(packed, f, positions=pos)
    M.masked_gqa_rope(xc, f)
    M.masked_gqa_rope(xu, f)
    torch.cuda.synchronize()
    assert torch.equal(packed[:, :, :1024], xc) and torch.equal(packed[:, :, 1024:], xu)


def test_rope_strided_view(M):
    # q laid out [B, L, H, D] and viewed as [B, H, L, D]: same bits as contiguous
    base = make_x(31, 2, 200, 16, 128, torch.bfloat16).cuda()  # [B, L, H, D]
    view = base.transpose(1, 2)
    cont = view.contiguous()
    f = inv_freq_table(128).cuda()
    M.masked_gqa_rope(view, f, interleaved=False)
    M.masked_gqa_rope(cont, f, interleaved=False)
    torch.cuda.synchronize()
    assert torch.equal(view, cont)


def test_rope_rejects_host_tensors_and_bad_tables(M):
    x = make_x(1, 1, 2, 8, 64, torch.bfloat16)
    with pytest.raises(ValueError):
        M.masked_gqa_rope(x, inv_freq_table(64))
    with pytest.raises(ValueError):
        M.masked_gqa_rope(x.cuda(), inv_freq_table(32).cuda())


def test_reduced_sincos_error_bound(M):
    """The rotation's sine and cosine (reduction by 2 pi, then the MUFU unit)
    against fp64 over the angles of positions up to 32768: rotating (1, 0) by
    theta gives (cos theta, sin theta) of the fp32 angle exactly as computed."""
    g = torch.Generator().manual_seed(77)
    L = 4096
    x = torch.zeros(1, 1, L, 2, dtype=torch.float32)
    x[..., 0] = 1.0
    pos = torch.randint(0, 32768, (1, L), generator=g, dtype=torch.int32)
    f = torch.tensor([0.99], dtype=torch.float32)
    xd = x.cuda()
    M.masked_gqa_rope(xd, f.cuda(), positions=pos.cuda(), interleaved=True)
    torch.cuda.synchronize()
    theta = (pos.to(torch.float32) * f[0]).double()[0]   # the fp32 product, widened
    got = xd.cpu().double()[0, 0]
    err = torch.maximum((got[:, 0] - torch.cos(theta)).abs(), (got[:, 1] - torch.sin(theta)).abs())
    assert float(err.max()) <= 1e-6, float(err.max())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("rot", [128, 64, 20])
def test_rope_vector_and_scalar_paths_agree(M, oracle_mod, dtype, interleaved, rot):
    """16-byte-aligned rows take the vector kernel, others the per-pair one:
    the same bits either way (a view one element into a padded buffer is not
    16-byte aligned; rot_dim 20 is not whole vectors and always takes the
    per-pair kernel)."""
    B, H, L, D, heads = 2, 6, 333, 128, 5
    x = make_x(51 + rot, B, H, L, D, dtype)
    f = inv_freq_table(rot)
    g = torch.Generator().manual_seed(8)
    pos = torch.randint(0, 8192, (B, L), generator=g, dtype=torch.int32)
    pad = torch.zeros(B, H, L, D + 8, dtype=dtype)
    pad[..., 1:D + 1] = x
    a, p = x.cuda(), pad.cuda()
    view = p[..., 1:D + 1]
    for t in (a, view):
        M.masked_gqa_rope(t, f.cuda(), positions=pos.cuda(), rot_dim=rot, heads=heads,
                          interleaved=interleaved)
    torch.cuda.synchronize()
    assert torch.equal(a.cpu(), view.cpu())
    assert torch.equal(p[..., 0].cpu(), pad[..., 0]) and torch.equal(p[..., D + 1:].cpu(), pad[..., D + 1:])
    ref = oracle_mod.rope(x, inv_freq=f, positions=pos, rot_dim=rot, heads=heads, interleaved=interleaved)
    assert_close_to_oracle(a, ref, dtype, f"rope rot {rot}")


PAIR_CASES = [  # q shape, k shape, rot_dim, q_heads, k_heads, q norm, k norm, k as a strided view
    ((2, 16, 1024, 128), (2, 8, 1024, 128), 128, 16, 8, False, False, False),  # one vector launch
    ((2, 16, 300, 128), (2, 8, 300, 128), 64, 16, 8, True, True, False),       # one norm launch
    ((1, 4, 77, 64), (1, 2, 77, 64), 64, 4, 2, True, False, False),            # norm and vector: two
    ((1, 4, 77, 64), (1, 2, 77, 66), 64, 3, 2, False, False, True),            # vector and scalar: two
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "x".join(map(str, c[0] + c[1])) + f"_{c[5]}{c[6]}{c[7]}")
def test_rope_pair_equals_two_calls(M, dtype, interleaved, case):
    """q and k in one launch (or two, when they take different kernels) give
    the bits of masked_gqa_rope on q followed by masked_gqa_rope on k."""
    qs, ks, rot, qh, kh, qn, kn, kview = case
    f = inv_freq_table(rot).cuda()
    g = torch.Generator().manual_seed(sum(qs) + sum(ks) + rot)
    pos = torch.randint(0, 4096, (qs[0], qs[2]), generator=g, dtype=torch.int32).cuda()
    q = make_x(11 + rot, *qs, dtype).cuda()
    kfull = make_x(12 + rot, *ks, dtype).cuda()
    k = kfull[..., :qs[3]] if kview else kfull  # a view whose rows are not 16-byte multiples
    wq = (torch.rand(qs[3], generator=g) + 0.5).cuda() if qn else None
    wk = (torch.rand(qs[3], generator=g) + 0.5).cuda() if kn else None
    q1, k1 = q.clone(), k.clone()
    M.masked_gqa_rope(q1, f, positions=pos, rot_dim=rot, heads=qh, interleaved=interleaved, norm_weight=wq)
    M.masked_gqa_rope(k1, f, positions=pos, rot_dim=rot, heads=kh, interleaved=interleaved, norm_weight=wk)
    M.masked_gqa_rope_pair(q, k, f, positions=pos, rot_dim=rot, q_heads=qh, k_heads=kh,
                           interleaved=interleaved, q_norm_weight=wq, k_norm_weight=wk)
    torch.cuda.synchronize()
    assert torch.equal(q, q1) and torch.equal(k, k1)
    if kview:  # the features past the view are untouched
        assert torch.equal(kfull[..., qs[3]:], make_x(12 + rot, *ks, dtype).cuda()[..., qs[3]:])


def test_rope_pair_overlapping_tensors_rotate_in_turn(M):
    """When q and k share elements the pair call rotates them one after the
    other, as two calls would (here: the same tensor, rotated twice)."""
    f = inv_freq_table(64).cuda()
    x = make_x(21, 1, 4, 100, 64, torch.bfloat16).cuda()
    ref = x.clone()
    M.masked_gqa_rope(ref, f)
    M.masked_gqa_rope(ref, f)
    M.masked_gqa_rope_pair(x, x, f)
    torch.cuda.synchronize()
    assert torch.equal(x, ref)


def test_rope_pair_rejects_mixed_dtypes_and_bad_args(M):
    f = inv_freq_table(64).cuda()
    q = make_x(1, 1, 2, 8, 64, torch.bfloat16).cuda()
    k = make_x(2, 1, 2, 8, 64, torch.float16).cuda()
    before = q.clone()
    with pytest.raises(M.MgqaError):
        M.masked_gqa_rope_pair(q, k, f)
    with pytest.raises(M.MgqaError):
        M.masked_gqa_rope_pair(q, q.clone(), f, k_heads=3)  # heads > H
    torch.cuda.synchronize()
    assert torch.equal(q, before)  # nothing was enqueued
