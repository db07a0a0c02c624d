"""The debug library (libmgqa_debug.so: the product sources built with
device-side bounds checks, event counters and an injectable pipeline stall).

* Its bounds checks stay silent on valid calls of every kernel, and its
  results equal the product library's bit for bit.
* Failure detection without a GPU fault: with the tensor-core prefill's load
  pipeline stalled on purpose (the producer issues no load from a given key
  tile on) and the wait limit cut to a few milliseconds, the consumers' bounded
  waits give up, the call reports MGQA_ERR_TIMEOUT in its device error word,
  the kernel returns, and the next normal call on the same stream is correct.
  Nothing here traps, faults or waits without a limit: every copy issued before
  the stall lands before its CTA exits and every MMA issued completes before
  the tensor memory is freed (the same failure path is run as a discrete-event
  model on the CPU in test_protocol_cpu.py)."""
import ctypes

import pytest
import torch

import workloads as W
from _util import assert_close_to_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import masked_gqa_attention_gb300 as M
    M.build_library()
    Ld = M.debug_lib()
    assert Ld.mgqa_debug_reset() == M.MGQA_OK
    yield M
    Ld.mgqa_debug_reset()


def _prefill(L, M, d, wl, err):
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device="cuda")
    a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, lse=lse, dev_error=err,
                    mask_bits=d["mask_bits"], kv_len=d["kv_len"], seg_q=d["seg_q"],
                    seg_k=d["seg_k"], causal=wl.causal)
    st = L.masked_gqa_attn_prefill(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == M.MGQA_OK, L.mgqa_last_error_detail()
    return out, lse


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("mask", ["none", "bits", "kvlen", "segment", "causal"])
def test_debug_prefill_checks_stay_silent_and_match(M, dtype, mask):
    wl = W.random_case(40 + len(mask), 2, 8, 2, 300, 700, 128 if dtype != torch.float32 else 64,
                       dtype=dtype, mask=mask)
    d = to_device(wl)
    outs = []
    for L in (M.lib(), M.debug_lib()):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(_prefill(L, M, d, wl, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error {int(err.item())}"
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("variant", ["full", "span"])
def test_debug_decode_checks_stay_silent_and_match(M, variant):
    wl = W.static_cache_decode(seed=61, variant=variant, B=4, capacity=3000, lo=1, hi=3000)
    d = to_device(wl)
    masks = {n: d[n] for n in ("mask_bits", "kv_len", "seg_q", "seg_k")}
    outs = []
    for L in (M.lib(), M.debug_lib()):
        out = torch.full_like(d["q"], float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = M.new_decode_workspace(d["q"], d["k"], d["v"], **masks)
        a = M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, dev_error=err, **masks)
        st = L.masked_gqa_attn_decode(ctypes.byref(a), ws.data_ptr(), ws.numel(),
                                      torch.cuda.current_stream().cuda_stream)
        assert st == M.MGQA_OK, L.mgqa_last_error_detail()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("stall_at", [1, 2])
@pytest.mark.parametrize("case", [(1, 2, 1, 640, 128), (1, 4, 4, 512, 64)],
                         ids=lambda c: "x".join(map(str, c)))
def test_stalled_pipeline_times_out_and_recovers(M, oracle_mod, stall_at, case):
    B, Hq, Hkv, L, D = case
    wl = W.random_case(3 + stall_at, B, Hq, Hkv, L, L, D, dtype=torch.bfloat16, mask="none")
    d = to_device(wl)
    Ld = M.debug_lib()
    # every query tile has L/128 >= 4 non-empty key tiles, so the stall at
    # list entry 1 or 2 leaves the pipeline waiting for a tile that never comes
    assert Ld.mgqa_debug_inject_prefill_stall(stall_at, 5_000_000) == M.MGQA_OK
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        _prefill(Ld, M, d, wl, err)
        torch.cuda.synchronize()
    finally:
        assert Ld.mgqa_debug_reset() == M.MGQA_OK
    assert int(err.item()) == M.MGQA_ERR_TIMEOUT
    # the context is healthy: the next normal call on the same stream is right
    err.zero_()
    out, _ = _prefill(Ld, M, d, wl, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _, _ = oracle_mod.attention(wl.q, wl.k, wl.v, scale=wl.scale)
    assert_close_to_oracle(out, ref, torch.bfloat16, "after the stall")
    out2, _ = _prefill(M.lib(), M, d, wl, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and torch.equal(out, out2)


def test_stall_arguments_are_checked(M):
    Ld = M.debug_lib()
    assert Ld.mgqa_debug_inject_prefill_stall(0, 1000) == M.MGQA_ERR_INVALID_ARG
    assert Ld.mgqa_debug_inject_prefill_stall(1, 0) == M.MGQA_ERR_INVALID_ARG
    assert Ld.mgqa_debug_inject_prefill_stall(-1, 0) == M.MGQA_OK
    buf = (ctypes.c_uint64 * 8)()
    assert Ld.mgqa_debug_counters(buf, 8) == M.MGQA_ERR_INVALID_ARG


def _timeline(fn, n):
    buf = (ctypes.c_uint64 * (n * 16))()
    assert fn(buf, n) == 0
    import numpy as np
    return np.array(buf, dtype=np.uint64).reshape(n, 16).astype(np.int64)


def test_phase_timelines_are_ordered_and_cleared(M):
    """The debug timelines (test equipment for finding where a kernel's time
    goes): every CTA that ran records its phases in order on one SM clock, and
    reading clears the record."""
    Ld = M.debug_lib()
    h = torch.cuda.current_stream().cuda_stream
    # prefill: the padded-CFG shape (8 query tiles x 8 head pairs x 2 rows)
    wl = W.padded_cfg(variant="kvlen")
    d = to_device(wl)
    _timeline(Ld.mgqa_debug_prefill_timeline, 1024)  # clear
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _prefill(Ld, M, d, wl, err)
    torch.cuda.synchronize()
    t = _timeline(Ld.mgqa_debug_prefill_timeline, 128)
    # pairs ordered by causality (same thread, or an issue and its completion)
    for k0, k1 in ((0, 1), (1, 9), (9, 11), (11, 12), (12, 2), (1, 3), (1, 10), (10, 4), (4, 5),
                   (5, 6), (6, 7)):
        assert (t[:, k1] >= t[:, k0]).all(), (k0, k1)
    assert (t[:, 14] >= t[:, 13]).all() and (t[:, 0] > 0).all()
    assert (_timeline(Ld.mgqa_debug_prefill_timeline, 128) == 0).all()
    # per-tile trace of the first CTAs (8 non-empty key tiles each in row 0)
    import numpy as np
    buf = (ctypes.c_uint64 * (4 * 64 * 18))()
    assert Ld.mgqa_debug_prefill_trace(buf, 4) == 0  # clear
    _prefill(Ld, M, d, wl, err)
    torch.cuda.synchronize()
    assert Ld.mgqa_debug_prefill_trace(buf, 4) == 0
    tr = np.array(buf, dtype=np.uint64).reshape(4, 64, 18).astype(np.int64)
    nk = 8
    # (key tile 0's loads go out before the producer loop: no issue stamps)
    assert (tr[:, :nk, :16] > 0).all() and (tr[:, 1:nk, 16:] > 0).all() and (tr[:, nk:, :] == 0).all()
    for t in range(2):
        e = tr[:, :nk]
        # same thread, or an MMA commit before the completion the softmax sees
        assert (e[..., 2 * t] <= e[..., 2 * t + 1]).all() and (e[..., 4 + 2 * t] <= e[..., 5 + 2 * t]).all()
        assert (e[..., 2 * t + 1] <= e[..., 8 + 4 * t]).all() and (e[..., 8 + 4 * t] <= e[..., 10 + 4 * t]).all()
        assert (e[..., 8 + 4 * t] <= e[..., 9 + 4 * t]).all()
    assert Ld.mgqa_debug_prefill_trace(buf, 4) == 0
    assert (np.array(buf, dtype=np.uint64) == 0).all()
    # decode: the static-cache shape (16 splits x 2 head groups x 8 requests)
    wd = W.static_cache_decode(variant="span")
    dd = to_device(wd)
    out = torch.empty_like(dd["q"])
    a = M.make_args(dd["q"], dd["k"], dd["v"], out, scale=wd.scale, kv_len=dd["kv_len"])
    _timeline(Ld.mgqa_debug_decode_timeline, 256)
    assert Ld.masked_gqa_attn_decode(ctypes.byref(a), None, 0, h) == 0
    torch.cuda.synchronize()
    t = _timeline(Ld.mgqa_debug_decode_timeline, 256)
    ran = t[:, 3] > 0  # CTAs with at least one chunk
    for k0, k1 in ((0, 1), (1, 2), (5, 6), (6, 7), (7, 8)):
        assert (t[:, k1] >= t[:, k0]).all(), (k0, k1)
    for k0, k1 in ((2, 3), (3, 4), (4, 5)):
        assert (t[ran, k1] >= t[ran, k0]).all(), (k0, k1)
    assert ran.any() and (_timeline(Ld.mgqa_debug_decode_timeline, 256) == 0).all()
