"""Shared helpers for the parity tests (comparison against the fp64 oracle)."""
import numpy as np
import torch

# bf16 I/O with fp32 accumulation: max abs <= 2e-2 and mean abs <= 2e-3 over all
# outputs; fp32 I/O: max abs error / max |oracle| <= 1e-5.
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
FP32_REL = 1e-5


def to_device(wl, device="cuda"):
    d = {}
    for name in ("q", "k", "v", "mask_bits", "kv_len", "seg_q", "seg_k"):
        t = getattr(wl, name)
        d[name] = None if t is None else t.to(device)
    return d


def assert_close_to_oracle(out_gpu, ref, dtype, what=""):
    got = out_gpu.detach().to("cpu", torch.float64).numpy()
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    # fp16 I/O is held to the bf16 bounds (its rounding is finer than bf16's)
    if dtype == torch.float32:
        rel = err.max() / max(np.abs(ref).max(), 1e-6)
        assert rel <= FP32_REL, f"{what}: fp32 relative error {rel:.3e} > {FP32_REL}"
        return dict(rel=float(rel))
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, \
        f"{what}: bf16 max abs {mx:.3e} (<= {BF16_MAX_ABS}), mean abs {mean:.3e} (<= {BF16_MEAN_ABS})"
    return dict(max_abs=mx, mean_abs=mean)


def assert_lse_close(lse_gpu, ref_lse, tol):
    got = lse_gpu.detach().to("cpu", torch.float64).numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got), fin), "LSE finiteness differs"
    assert np.all(got[~fin] == -np.inf)
    if fin.any():
        err = np.abs(got[fin] - ref_lse[fin]).max()
        assert err <= tol, f"LSE error {err:.3e} > {tol}"
