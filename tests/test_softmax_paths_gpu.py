"""Parity of the tensor-core prefill's online softmax on the two paths that
N(0,1) inputs never reach, against the fp64 oracle:

* the lazy rescale of the running output, taken only when a row's maximum
  grows by more than 2^8 between key tiles (real attention logits span that
  much: the VoxCPM page, "Upstream-identical practice", attention bullet,
  asks for SDPA's result at any scale);
* a negative softmax scale (the running maximum of scaled scores is then the
  minimum of the raw ones).

Each rescale case also runs through the debug library, whose counter of
rescale events must be non-zero (the branch really ran) and whose output
must equal the product library's bit for bit (same arithmetic)."""
import ctypes

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


def _call(L, M, d, wl, out, lse, err):
    a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, lse=lse, dev_error=err,
                    mask_bits=d["mask_bits"], kv_len=d["kv_len"], seg_q=d["seg_q"],
                    seg_k=d["seg_k"], causal=wl.causal)
    st = L.masked_gqa_attn_prefill(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == M.MGQA_OK, L.mgqa_last_error_detail()


def run(M, wl, library=None):
    L = library or M.lib()
    d = to_device(wl)
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _call(L, M, d, wl, out, lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error {int(err.item())}"
    return out, lse


def counters(M):
    Ld = M.debug_lib()
    buf = (ctypes.c_uint64 * M.DEBUG_NUM_COUNTERS)()
    assert Ld.mgqa_debug_counters(buf, M.DEBUG_NUM_COUNTERS) == M.MGQA_OK
    return list(buf)


def check_against_oracle(oracle_mod, wl, out, lse, what):
    ref, ref_lse, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale, **wl.masks())
    assert_close_to_oracle(out, ref, wl.q.dtype, what)
    assert_lse_close(lse, ref_lse, 2e-3 * max(1.0, float(abs(ref_lse[abs(ref_lse) < 1e30]).max()) / 8))


def rescale_events(M, wl):
    """Run wl through the debug library; returns (out, lse, rescale events)."""
    Ld = M.debug_lib()
    assert Ld.mgqa_debug_reset() == M.MGQA_OK
    out, lse = run(M, wl, library=Ld)
    c = counters(M)
    assert c[1] > 0, "the debug counters saw no tile at all"
    return out, lse, c[0]


SHAPES = [
    # B, Hq, Hkv, L, D: the padded-CFG heads at a ragged length, the DiT heads, head dim 64
    (2, 16, 8, 1000, 128),
    (1, 16, 4, 1300, 128),
    (2, 4, 2, 700, 64),
    (1, 2, 2, 513, 128),  # one head per KV head: single-head CTAs
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mask", ["none", "bits", "segment"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda c: "x".join(map(str, c)))
def test_rescale_branch_matches_oracle(M, oracle_mod, dtype, mask, shape):
    wl = W.growing_scores(sum(shape) + len(mask), *shape, dtype=dtype, mask=mask)
    out, lse = run(M, wl)
    check_against_oracle(oracle_mod, wl, out, lse, f"rescale {mask} {shape}")
    out_d, lse_d, events = rescale_events(M, wl)
    assert events > 0, "the rescale branch never ran"
    assert torch.equal(out, out_d) and torch.equal(lse, lse_d)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rescale_after_a_lone_low_key(M, oracle_mod, dtype):
    """The second segment starts at key 127: its rows see one near-zero score
    in their first (partial) tile, then scores far higher in the next tiles."""
    wl = W.late_spike(77, 2, 8, 4, 900, 128, dtype=dtype)
    out, lse = run(M, wl)
    check_against_oracle(oracle_mod, wl, out, lse, "late spike")
    out_d, lse_d, events = rescale_events(M, wl)
    assert events > 0
    assert torch.equal(out, out_d) and torch.equal(lse, lse_d)


def test_plain_inputs_never_rescale(M):
    """Control for the counter: N(0,1) inputs at scale 1/sqrt(D) stay within
    2^8 of their first tile's maximum."""
    wl = W.random_case(5, 2, 8, 4, 1024, 1024, 128, dtype=torch.bfloat16, mask="none")
    _, _, events = rescale_events(M, wl)
    assert events == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mask", ["none", "bits", "kvlen", "segment", "causal"])
@pytest.mark.parametrize("shape", [(2, 8, 4, 600, 128), (1, 4, 2, 333, 64), (1, 2, 2, 256, 128)],
                         ids=lambda c: "x".join(map(str, c)))
def test_negative_scale_matches_oracle(M, oracle_mod, dtype, mask, shape):
    B, Hq, Hkv, L, D = shape
    wl = W.random_case(B + Hq + L + 11 * len(mask), B, Hq, Hkv, L, L, D, dtype=dtype, mask=mask)
    wl.scale = -wl.scale
    out, lse = run(M, wl)
    check_against_oracle(oracle_mod, wl, out, lse, f"negative scale {mask} {shape}")


@pytest.mark.parametrize("mask", ["none", "bits"])
def test_negative_scale_with_rescale(M, oracle_mod, mask):
    wl = W.growing_scores(31, 2, 8, 4, 900, 128, dtype=torch.bfloat16, mask=mask)
    wl.scale = -wl.scale
    out, lse = run(M, wl)
    check_against_oracle(oracle_mod, wl, out, lse, f"negative scale, growing {mask}")
    out_d, lse_d, events = rescale_events(M, wl)
    assert events > 0
    assert torch.equal(out, out_d) and torch.equal(lse, lse_d)
