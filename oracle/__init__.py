"""Oracle for masked grouped-query attention (fp64, CPU).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The product library
never links or calls it, and it imports nothing from the product package.

The arithmetic lives in ``mgqa_oracle.c`` (plain fp64 loops, OpenMP over
(batch, query head, query row)); this module only compiles it and converts
arrays. What it computes, with the passages it follows:

* VoxCPM page, "Upstream-identical practice", attention bullet: SDPA with
  ``enable_gqa`` on contiguous tensors, bidirectional, and cache decode under
  an explicit boolean mask whose masked slots add exact zeros;
* OmniVoice page, "Upstream-identical practice", attention-mask bullet: a
  full 4D boolean mask, not causal, KV heads repeated to the query heads;
* OmniVoice page, "Memory & speed", packed_guidance paragraph: a
  block-diagonal mask, each block equal to its run alone;
* VoxCPM page, "Upstream-identical practice", attention bullet: causal
  attention at prefill (query rows = the last Lq of the Lk positions);
* RMS normalisation of head vectors (``rms_norm``): OmniVoice page, "Parity
  results" (q and k normalised separately before the rotation);
* rotary position embedding (``rope``): F5-TTS page (interleaved pairs, on
  the first pe_attn_head heads), OmniVoice page, "Parity results", and VoxCPM page, precision bullet (fp32 inverse
  frequencies, LongRoPE tables built in fp32), OmniVoice page, packed_guidance
  paragraph (positions restart per packed sequence).

Readings where the pages are silent (each also listed in the design notes):
query head h reads KV head ``h // (Hq // Hkv)``; mask ``True`` means "may
attend"; packed mask bits are least-significant-bit first in uint32 words; a
query row with no allowed key gives output 0 and LSE ``-inf``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mgqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmgqa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C source into a shared library (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.mgqa_oracle_attention
            P = ctypes.c_void_p
            I = ctypes.c_int
            f.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, P, I,
                          ctypes.c_double, P, P, I]
            f.restype = I
            g = lib.mgqa_oracle_rope
            g.argtypes = [P, I, I, I, I, P, P, I, I, I]
            g.restype = I
            n = lib.mgqa_oracle_rms_norm
            n.argtypes = [P, I, I, I, I, P, ctypes.c_double, I]
            n.restype = I
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact widening of bf16/fp32/fp64 input (torch tensor or array) to fp64."""
    if hasattr(x, "detach"):  # torch tensor: widen in torch (bf16 has no numpy dtype)
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.int32)


def _u32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = np.asarray(x)
    if a.dtype == np.int32:
        a = a.view(np.uint32)
    return np.ascontiguousarray(a, dtype=np.uint32)


def attention(q, k, v, *, scale: float, mask_bits=None, kv_len=None,
              seg_q=None, seg_k=None, causal: bool = False, threads: int = 0):
    """Masked GQA attention in fp64.

    q: [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D]; mask_bits: uint32
    [B, Lq, ceil(Lk/32)] (LSB-first, 1 = attend); kv_len: int32 [B];
    seg_q: int32 [B, Lq]; seg_k: int32 [B, Lk]; causal: key j only for query
    i with j <= i + Lk - Lq. Returns (out [B,Hq,Lq,D],
    lse [B,Hq,Lq], threads_used), all fp64 except the count.
    """
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, D = q64.shape
    Bk, Hkv, Lk, Dk = k64.shape
    if (Bk, Dk) != (B, D) or v64.shape != k64.shape:
        raise ValueError("shape mismatch between q, k and v")
    bits, kvl, sq, sk = _u32(mask_bits), _i32(kv_len), _i32(seg_q), _i32(seg_k)
    W = (Lk + 31) // 32
    if bits is not None and bits.shape != (B, Lq, W):
        raise ValueError(f"mask_bits must be [B, Lq, {W}] uint32")
    if kvl is not None and kvl.shape != (B,):
        raise ValueError("kv_len must be [B]")
    if (sq is None) != (sk is None):
        raise ValueError("seg_q and seg_k go together")
    if sq is not None and (sq.shape != (B, Lq) or sk.shape != (B, Lk)):
        raise ValueError("seg_q must be [B, Lq] and seg_k [B, Lk]")
    out = np.zeros((B, Hq, Lq, D), dtype=np.float64)
    lse = np.zeros((B, Hq, Lq), dtype=np.float64)

    def ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    used = _load().mgqa_oracle_attention(
        ptr(q64), ptr(k64), ptr(v64), B, Hq, Hkv, Lq, Lk, D,
        ptr(bits), ptr(kvl), ptr(sq), ptr(sk), int(bool(causal)), float(scale),
        ptr(out), ptr(lse), int(threads))
    if used < 0:
        raise ValueError("oracle rejected the shapes")
    return out, lse, used


def rope(x, *, inv_freq, positions=None, rot_dim=None, heads=None, interleaved=False):
    """Rotary position embedding in fp64 (see mgqa_oracle_rope in the C file).

    x: [B, H, L, D] (any float type, widened exactly); inv_freq: [rot_dim/2]
    fp32; positions: int32 [B, L] or None (position = row index); rot_dim:
    rotated features per head (default D); heads: rotated heads (default H).
    Returns the rotated copy as fp64.
    """
    x64 = _f64(x).copy()
    B, H, L, D = x64.shape
    rot_dim = D if rot_dim is None else int(rot_dim)
    heads = H if heads is None else int(heads)
    f = inv_freq.detach().cpu().numpy() if hasattr(inv_freq, "detach") else inv_freq
    f = np.ascontiguousarray(np.asarray(f), dtype=np.float32)
    if f.shape != (rot_dim // 2,):
        raise ValueError(f"inv_freq must be [{rot_dim // 2}] fp32")
    pos = _i32(positions)
    if pos is not None and pos.shape != (B, L):
        raise ValueError("positions must be [B, L] int32")
    rc = _load().mgqa_oracle_rope(
        x64.ctypes.data_as(ctypes.c_void_p), B, H, L, D,
        None if pos is None else pos.ctypes.data_as(ctypes.c_void_p),
        f.ctypes.data_as(ctypes.c_void_p), rot_dim, heads, int(bool(interleaved)))
    if rc != 0:
        raise ValueError("oracle rejected the rope arguments")
    return x64


def rms_norm(x, *, weight, eps=1e-6, heads=None):
    """RMS normalisation over the head dim, in fp64 (see mgqa_oracle_rms_norm):
    y = x / sqrt(mean(x^2) + eps) * weight, for heads h < `heads` (default all).

    x: [B, H, L, D] (any float type, widened exactly); weight: [D] fp32.
    Returns the normalised copy as fp64.
    """
    x64 = _f64(x).copy()
    B, H, L, D = x64.shape
    heads = H if heads is None else int(heads)
    w = weight.detach().cpu().numpy() if hasattr(weight, "detach") else weight
    w = np.ascontiguousarray(np.asarray(w), dtype=np.float32)
    if w.shape != (D,):
        raise ValueError(f"weight must be [{D}] fp32")
    rc = _load().mgqa_oracle_rms_norm(x64.ctypes.data_as(ctypes.c_void_p), B, H, L, D,
                                      w.ctypes.data_as(ctypes.c_void_p), float(eps), heads)
    if rc != 0:
        raise ValueError("oracle rejected the rms_norm arguments")
    return x64
