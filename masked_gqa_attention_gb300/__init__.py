"""Python binding of the masked GQA attention library (libmgqa.so, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/masked_gqa_attn.h``. PyTorch
is used for device memory and streams. There is no CPU path: calling into
the library without the built extension or without a CUDA device raises.

Entry points (same names as the C ABI):
  * :func:`masked_gqa_attn_prefill` -- bidirectional full-sequence attention
    under a packed-bit mask, per-row key lengths and/or segment ids;
  * :func:`masked_gqa_attn_decode` -- one query per row over a static KV
    cache, merged on chip (the ``workspace`` arguments are accepted and
    ignored).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from .build import LIB as _LIB_PATH
from .build import LIB_DEBUG as _LIB_DEBUG_PATH
from .build import build as build_library

__all__ = [
    "MGQA_OK", "MGQA_ERR_INVALID_ARG", "MGQA_ERR_UNSUPPORTED", "MGQA_ERR_CUDA",
    "MGQA_ERR_TIMEOUT", "MgqaError", "MgqaArgs", "lib", "make_args",
    "masked_gqa_attn_prefill", "masked_gqa_attn_decode",
    "masked_gqa_attn_decode_workspace_size", "new_decode_workspace", "build_library",
    "masked_gqa_attn_decode_static",
    "masked_gqa_attn_decode_append", "masked_gqa_pack_pair", "masked_gqa_unpack_pair",
    "debug_lib", "MGQA_ERR_DEVICE_CHECK", "MgqaQkRope", "make_qk_rope",
    "masked_gqa_attn_prefill_rope", "masked_gqa_attn_decode_append_rope", "masked_gqa_rope",
    "masked_gqa_rope_pair",
]

(MGQA_OK, MGQA_ERR_INVALID_ARG, MGQA_ERR_UNSUPPORTED, MGQA_ERR_CUDA, MGQA_ERR_TIMEOUT,
 MGQA_ERR_DEVICE_CHECK) = range(6)
MGQA_BF16, MGQA_FP32, MGQA_FP16 = 0, 1, 2

EXPORTED_SYMBOLS = (
    "masked_gqa_attn_prefill",
    "masked_gqa_attn_decode_workspace_size",
    "masked_gqa_attn_decode",
    "mgqa_status_string",
    "mgqa_last_error_detail",
    "mgqa_abi_version",
    "masked_gqa_attn_decode_static",
    "masked_gqa_attn_decode_append",
    "masked_gqa_pack_pair",
    "masked_gqa_unpack_pair",
    "masked_gqa_rope",
    "masked_gqa_attn_prefill_rope",
    "masked_gqa_attn_decode_append_rope",
    "masked_gqa_rope_pair",
)
# exported by the debug library only (include/masked_gqa_attn_debug.h)
DEBUG_SYMBOLS = (
    "mgqa_debug_counters",
    "mgqa_debug_reset",
    "mgqa_debug_inject_prefill_stall",
    "mgqa_debug_decode_timeline",
    "mgqa_debug_prefill_timeline",
    "mgqa_debug_prefill_trace",
)
DEBUG_NUM_COUNTERS = 4


class MgqaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"mgqa status {status}: {detail}")
        self.status = status
        self.detail = detail


class MgqaArgs(ctypes.Structure):
    """Mirror of ``mgqa_args`` in include/masked_gqa_attn.h."""
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("Lq", ctypes.c_int32), ("Lk", ctypes.c_int32), ("D", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("mask_bits", ctypes.c_void_p),
        ("mask_stride_b", ctypes.c_int64), ("mask_stride_q", ctypes.c_int64),
        ("kv_len", ctypes.c_void_p),
        ("seg_q", ctypes.c_void_p), ("seg_k", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("lse", ctypes.c_void_p),
        ("dev_error", ctypes.c_void_p),
        ("causal", ctypes.c_int32),
    ]


class MgqaRopeArgs(ctypes.Structure):
    """Mirror of ``mgqa_rope_args`` in include/masked_gqa_attn.h."""
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32), ("D", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("x_stride", ctypes.c_int64 * 3),
        ("positions", ctypes.c_void_p),
        ("inv_freq", ctypes.c_void_p),
        ("rot_dim", ctypes.c_int32), ("heads", ctypes.c_int32), ("interleaved", ctypes.c_int32),
        ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
    ]


class MgqaQkRope(ctypes.Structure):
    """Mirror of ``mgqa_qk_rope`` in include/masked_gqa_attn.h."""
    _fields_ = [
        ("inv_freq", ctypes.c_void_p), ("positions", ctypes.c_void_p),
        ("rot_dim", ctypes.c_int32), ("interleaved", ctypes.c_int32),
        ("q_heads", ctypes.c_int32), ("k_heads", ctypes.c_int32),
        ("q_norm_weight", ctypes.c_void_p), ("k_norm_weight", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
    ]


_lib = None
_lib_debug = None


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    """Argument and result types of the C ABI's entry points."""
    P = ctypes.c_void_p
    I64P = ctypes.POINTER(ctypes.c_int64)
    I32 = ctypes.c_int32
    L.masked_gqa_attn_prefill.argtypes = [ctypes.POINTER(MgqaArgs), P]
    L.masked_gqa_attn_prefill.restype = ctypes.c_int
    L.masked_gqa_attn_decode_workspace_size.argtypes = [ctypes.POINTER(MgqaArgs)]
    L.masked_gqa_attn_decode_workspace_size.restype = ctypes.c_size_t
    L.masked_gqa_attn_decode.argtypes = [ctypes.POINTER(MgqaArgs), P, ctypes.c_size_t, P]
    L.masked_gqa_attn_decode.restype = ctypes.c_int
    L.mgqa_status_string.argtypes = [ctypes.c_int]
    L.mgqa_status_string.restype = ctypes.c_char_p
    L.mgqa_last_error_detail.argtypes = []
    L.mgqa_last_error_detail.restype = ctypes.c_char_p
    L.masked_gqa_attn_decode_append.argtypes = [ctypes.POINTER(MgqaArgs), P, P, I64P, I64P, P, P,
                                                ctypes.c_size_t, P]
    L.masked_gqa_attn_decode_append.restype = ctypes.c_int
    L.masked_gqa_pack_pair.argtypes = [ctypes.c_int, I32, I32, I32, P, I64P, I32, P, I64P, I32,
                                       P, I64P, P, P]
    L.masked_gqa_pack_pair.restype = ctypes.c_int
    L.masked_gqa_unpack_pair.argtypes = [ctypes.c_int, I32, I32, I32, P, I64P, P, I64P, I32,
                                         P, I64P, I32, P]
    L.masked_gqa_unpack_pair.restype = ctypes.c_int
    L.masked_gqa_attn_decode_static.argtypes = [ctypes.POINTER(MgqaArgs), P]
    L.masked_gqa_attn_decode_static.restype = ctypes.c_int
    L.masked_gqa_rope.argtypes = [ctypes.POINTER(MgqaRopeArgs), P]
    L.masked_gqa_rope.restype = ctypes.c_int
    L.masked_gqa_rope_pair.argtypes = [ctypes.POINTER(MgqaRopeArgs), ctypes.POINTER(MgqaRopeArgs), P]
    L.masked_gqa_rope_pair.restype = ctypes.c_int
    L.mgqa_abi_version.argtypes = []
    L.mgqa_abi_version.restype = ctypes.c_int32
    L.masked_gqa_attn_prefill_rope.argtypes = [ctypes.POINTER(MgqaArgs), ctypes.POINTER(MgqaQkRope), P]
    L.masked_gqa_attn_prefill_rope.restype = ctypes.c_int
    L.masked_gqa_attn_decode_append_rope.argtypes = [ctypes.POINTER(MgqaArgs), P, P, I64P, I64P, P,
                                                     ctypes.POINTER(MgqaQkRope), P, ctypes.c_size_t, P]
    L.masked_gqa_attn_decode_append_rope.restype = ctypes.c_int
    return L


def lib() -> ctypes.CDLL:
    """Load libmgqa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmgqa.so is not built ({_LIB_PATH}); run build_library()")
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def debug_lib() -> ctypes.CDLL:
    """Load libmgqa_debug.so: the same entry points built with device-side
    bounds checks, event counters and an injectable pipeline stall, plus the
    mgqa_debug_* functions (test equipment; raises if it has not been built)."""
    global _lib_debug
    if _lib_debug is None:
        if not os.path.exists(_LIB_DEBUG_PATH):
            raise RuntimeError(f"libmgqa_debug.so is not built ({_LIB_DEBUG_PATH}); "
                               "run build_library()")
        L = _bind(ctypes.CDLL(_LIB_DEBUG_PATH))
        L.mgqa_debug_counters.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32]
        L.mgqa_debug_counters.restype = ctypes.c_int
        L.mgqa_debug_reset.argtypes = []
        L.mgqa_debug_reset.restype = ctypes.c_int
        L.mgqa_debug_inject_prefill_stall.argtypes = [ctypes.c_int32, ctypes.c_uint64]
        L.mgqa_debug_inject_prefill_stall.restype = ctypes.c_int
        L.mgqa_debug_decode_timeline.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32]
        L.mgqa_debug_decode_timeline.restype = ctypes.c_int
        L.mgqa_debug_prefill_timeline.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32]
        L.mgqa_debug_prefill_timeline.restype = ctypes.c_int
        L.mgqa_debug_prefill_trace.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32]
        L.mgqa_debug_prefill_trace.restype = ctypes.c_int
        _lib_debug = L
    return _lib_debug


def _check(status: int):
    if status != MGQA_OK:
        L = lib()
        detail = L.mgqa_last_error_detail().decode() or L.mgqa_status_string(status).decode()
        raise MgqaError(status, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    return t


def make_args(q, k, v, out, *, scale=None, mask_bits=None, kv_len=None, seg_q=None,
              seg_k=None, lse=None, dev_error=None, causal=False) -> MgqaArgs:
    """Fill an MgqaArgs from tensors: q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D], out like q.

    mask_bits: int32/uint32 words [B, Lq, W] (or [B, 1, W] / [1, Lq, W] with
    stride 0 broadcast), W >= ceil(Lk/32); kv_len int32 [B]; seg_q int32 [B, Lq];
    seg_k int32 [B, Lk]; lse fp32 [B, Hq, Lq] contiguous; dev_error int32 [1];
    causal: key j only for query i with j <= i + Lk - Lq.
    Tensors are passed by pointer; no copy is made.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _dev(t, name)
        if t.dim() != 4 or t.stride(3) != 1:
            raise ValueError(f"{name} must be 4-D with a unit-stride head dim")
    if q.dtype == torch.bfloat16:
        dt = MGQA_BF16
    elif q.dtype == torch.float32:
        dt = MGQA_FP32
    elif q.dtype == torch.float16:
        dt = MGQA_FP16
    else:
        raise ValueError("q/k/v must be bfloat16, float16 or float32")
    for name, t in (("k", k), ("v", v), ("out", out)):
        if t.dtype != q.dtype:
            raise ValueError(f"{name} dtype differs from q")
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch among q, k, v, out")
    a = MgqaArgs()
    a.dtype = dt
    a.B, a.Hq, a.Hkv, a.Lq, a.Lk, a.D = B, Hq, Hkv, Lq, Lk, D
    a.q, a.k, a.v, a.out = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr()
    for fld, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", out)):
        getattr(a, fld)[:] = [t.stride(0), t.stride(1), t.stride(2)]
    if mask_bits is not None:
        _dev(mask_bits, "mask_bits")
        if mask_bits.dtype not in (torch.int32, torch.uint32) or mask_bits.dim() != 3:
            raise ValueError("mask_bits must be 3-D int32/uint32 words")
        if mask_bits.stride(2) != 1:
            raise ValueError("mask_bits words must be contiguous along keys")
        if (mask_bits.shape[0] not in (1, B) or mask_bits.shape[1] not in (1, Lq)
                or mask_bits.shape[2] < (Lk + 31) // 32):
            raise ValueError(f"mask_bits must be [B or 1, Lq or 1, >= {(Lk + 31) // 32}] words")
        a.mask_bits = mask_bits.data_ptr()
        a.mask_stride_b = mask_bits.stride(0) if mask_bits.shape[0] > 1 else 0
        a.mask_stride_q = mask_bits.stride(1) if mask_bits.shape[1] > 1 else 0
    a.kv_len = _ptr(_dev(kv_len, "kv_len", torch.int32))
    if (seg_q is None) != (seg_k is None):
        raise ValueError("seg_q and seg_k go together")
    if seg_q is not None:
        for name, t, L in (("seg_q", seg_q, Lq), ("seg_k", seg_k, Lk)):
            _dev(t, name, torch.int32)
            if tuple(t.shape) != (B, L) or not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous int32 [B, {L}]")
        a.seg_q, a.seg_k = seg_q.data_ptr(), seg_k.data_ptr()
    a.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    if lse is not None:
        _dev(lse, "lse", torch.float32)
        if tuple(lse.shape) != (B, Hq, Lq) or not lse.is_contiguous():
            raise ValueError("lse must be contiguous fp32 [B, Hq, Lq]")
        a.lse = lse.data_ptr()
    a.dev_error = _ptr(_dev(dev_error, "dev_error", torch.int32))
    a.causal = 1 if causal else 0
    return a


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def masked_gqa_attn_prefill(q, k, v, out=None, *, scale=None, mask_bits=None, kv_len=None,
                            seg_q=None, seg_k=None, lse=None, dev_error=None, causal=False,
                            stream=None):
    """Masked GQA attention over full sequences (bidirectional unless causal); returns out."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k, v, out, scale=scale, mask_bits=mask_bits, kv_len=kv_len, seg_q=seg_q,
                  seg_k=seg_k, lse=lse, dev_error=dev_error, causal=causal)
    _check(lib().masked_gqa_attn_prefill(ctypes.byref(a), _stream_handle(stream)))
    return out


def _workspace(ws):
    """(pointer, bytes) of an optional decode workspace (ignored by the kernel)."""
    if ws is None:
        return None, 0
    _dev(ws, "workspace")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def masked_gqa_attn_decode_workspace_size(q, k, v, **masks) -> int:
    out = q  # shape/dtype stand-in; the library only reads the sizes
    a = make_args(q, k, v, out, **masks)
    n = lib().masked_gqa_attn_decode_workspace_size(ctypes.byref(a))
    if n == 0:
        _check(MGQA_ERR_INVALID_ARG)
    return int(n)


def new_decode_workspace(q, k, v, **masks) -> torch.Tensor:
    """A workspace tensor (uint8) of the nominal size for these decode
    arguments; the kernel never touches it (kept for earlier callers)."""
    n = masked_gqa_attn_decode_workspace_size(q, k, v, **masks)
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def masked_gqa_attn_decode(q, k, v, out=None, *, workspace: Optional[torch.Tensor] = None, scale=None,
                           mask_bits=None, kv_len=None, seg_q=None, seg_k=None, lse=None,
                           dev_error=None, stream=None):
    """One query per row (q [B, Hq, 1, D]) over a static cache k/v [B, Hkv, Lk, D]."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k, v, out, scale=scale, mask_bits=mask_bits, kv_len=kv_len, seg_q=seg_q,
                  seg_k=seg_k, lse=lse, dev_error=dev_error)
    wp, wn = _workspace(workspace)
    _check(lib().masked_gqa_attn_decode(ctypes.byref(a), wp, wn, _stream_handle(stream)))
    return out


def masked_gqa_attn_decode_static(q, k, v, out=None, *, scale=None, mask_bits=None, kv_len=None,
                                  seg_q=None, seg_k=None, lse=None, dev_error=None, stream=None):
    """masked_gqa_attn_decode without a workspace argument, for callers that
    may not allocate device memory: the kernel's scratch is its own on-chip
    shared memory, so nothing is allocated and calls do not share state."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k, v, out, scale=scale, mask_bits=mask_bits, kv_len=kv_len, seg_q=seg_q,
                  seg_k=seg_k, lse=lse, dev_error=dev_error)
    _check(lib().masked_gqa_attn_decode_static(ctypes.byref(a), _stream_handle(stream)))
    return out


def masked_gqa_attn_decode_append(q, k_cache, v_cache, k_new, v_new, kv_len, out=None, *,
                                  workspace: Optional[torch.Tensor] = None, kv_len_out=None,
                                  scale=None, lse=None,
                                  dev_error=None, stream=None):
    """One decode step fused with its cache append: k_new/v_new [B, Hkv, 1, D]
    go to slot kv_len[b] of k_cache/v_cache [B, Hkv, Lk, D] (written in place),
    then q [B, Hq, 1, D] attends over slots 0..kv_len[b]; kv_len_out (int32 [B],
    optional, not kv_len itself) receives kv_len + 1."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k_cache, v_cache, out, scale=scale, kv_len=kv_len, lse=lse,
                  dev_error=dev_error)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _dev(t, name, q.dtype)
        if t.dim() != 4 or t.shape[2] != 1 or t.stride(3) != 1:
            raise ValueError(f"{name} must be [B, Hkv, 1, D] with a unit-stride head dim")
    ks = (ctypes.c_int64 * 2)(k_new.stride(0), k_new.stride(1))
    vs = (ctypes.c_int64 * 2)(v_new.stride(0), v_new.stride(1))
    wp, wn = _workspace(workspace)
    _check(lib().masked_gqa_attn_decode_append(
        ctypes.byref(a), k_new.data_ptr(), v_new.data_ptr(), ks, vs,
        _ptr(_dev(kv_len_out, "kv_len_out", torch.int32)), wp, wn, _stream_handle(stream)))
    return out


def _dtype_code(t):
    return {torch.bfloat16: MGQA_BF16, torch.float16: MGQA_FP16, torch.float32: MGQA_FP32}[t.dtype]


def _st3(t):
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def masked_gqa_pack_pair(a, b, *, stream=None):
    """Pack two sequences [B, H, La, D] and [B, H, Lb, D] into one block-diagonal
    row [B, H, La + Lb, D]; returns (packed, seg) with seg int32 [B, La + Lb]
    (0 for a's positions, 1 for b's) for seg_q / seg_k."""
    for name, t in (("a", a), ("b", b)):
        _dev(t, name, a.dtype)
    B, H, La, D = a.shape
    Lb = b.shape[2]
    packed = torch.empty((B, H, La + Lb, D), dtype=a.dtype, device=a.device)
    seg = torch.empty((B, La + Lb), dtype=torch.int32, device=a.device)
    _check(lib().masked_gqa_pack_pair(_dtype_code(a), B, H, D, a.data_ptr(), _st3(a), La,
                                      b.data_ptr(), _st3(b), Lb, packed.data_ptr(),
                                      _st3(packed), seg.data_ptr(), _stream_handle(stream)))
    return packed, seg


def masked_gqa_unpack_pair(packed, La, *, stream=None):
    """Split a packed [B, H, La + Lb, D] output into ([B, H, La, D], [B, H, Lb, D])."""
    _dev(packed, "packed")
    B, H, L, D = packed.shape
    a = torch.empty((B, H, La, D), dtype=packed.dtype, device=packed.device)
    b = torch.empty((B, H, L - La, D), dtype=packed.dtype, device=packed.device)
    _check(lib().masked_gqa_unpack_pair(_dtype_code(packed), B, H, D, packed.data_ptr(),
                                        _st3(packed), a.data_ptr(), _st3(a), La, b.data_ptr(),
                                        _st3(b), L - La, _stream_handle(stream)))
    return a, b


def _rope_args(x, inv_freq, positions, rot_dim, heads, interleaved, norm_weight, norm_eps):
    _dev(x, "x")
    B, H, L, D = x.shape
    if x.stride(3) != 1:
        raise ValueError("x must have a contiguous head dimension")
    rot_dim = D if rot_dim is None else int(rot_dim)
    heads = H if heads is None else int(heads)
    _dev(inv_freq, "inv_freq", torch.float32)
    if not inv_freq.is_contiguous() or inv_freq.numel() != rot_dim // 2:
        raise ValueError(f"inv_freq must be a contiguous fp32 tensor of {rot_dim // 2} values")
    if positions is not None:
        _dev(positions, "positions", torch.int32)
        if tuple(positions.shape) != (B, L) or not positions.is_contiguous():
            raise ValueError("positions must be a contiguous int32 [B, L] tensor")
    a = MgqaRopeArgs()
    a.dtype = _dtype_code(x)
    a.B, a.H, a.L, a.D = B, H, L, D
    a.x = x.data_ptr()
    a.x_stride = _st3(x)
    a.positions = _ptr(positions)
    a.inv_freq = inv_freq.data_ptr()
    a.rot_dim, a.heads, a.interleaved = rot_dim, heads, int(bool(interleaved))
    if norm_weight is not None:
        _dev(norm_weight, "norm_weight", torch.float32)
        if not norm_weight.is_contiguous() or norm_weight.numel() != D:
            raise ValueError(f"norm_weight must be a contiguous fp32 tensor of {D} values")
        a.norm_weight = norm_weight.data_ptr()
        a.norm_eps = float(norm_eps)
    return a


def masked_gqa_rope(x, inv_freq, *, positions=None, rot_dim=None, heads=None, interleaved=False,
                    norm_weight=None, norm_eps=1e-6, stream=None):
    """Rotate x [B, H, L, D] (bf16, fp16 or fp32, head dim contiguous) in place by
    rotary position embedding and return it: theta = fl32(position * inv_freq[i])
    for pair i of the first rot_dim features (default D) of the first `heads`
    heads (default H); positions int32 [B, L] (default: the row index);
    inv_freq fp32 [rot_dim / 2]; interleaved pairs (2i, 2i+1) or half-split
    pairs (i, i + rot_dim/2). norm_weight (fp32 [D], optional): RMS-normalise
    each rotated head vector over its D features before the rotation."""
    a = _rope_args(x, inv_freq, positions, rot_dim, heads, interleaved, norm_weight, norm_eps)
    _check(lib().masked_gqa_rope(ctypes.byref(a), _stream_handle(stream)))
    return x


def masked_gqa_rope_pair(q, k, inv_freq, *, positions=None, rot_dim=None, q_heads=None,
                         k_heads=None, interleaved=False, q_norm_weight=None, k_norm_weight=None,
                         norm_eps=1e-6, stream=None):
    """Rotate q and k (same dtype; [B, H, L, D] each, head dim contiguous) in
    place with one launch, as masked_gqa_rope(q, ...) then masked_gqa_rope(k,
    ...) would (same bits): the same table and positions, each its own head
    count (default all) and optional norm weight. Returns (q, k)."""
    aq = _rope_args(q, inv_freq, positions, rot_dim, q_heads, interleaved, q_norm_weight, norm_eps)
    ak = _rope_args(k, inv_freq, positions, rot_dim, k_heads, interleaved, k_norm_weight, norm_eps)
    _check(lib().masked_gqa_rope_pair(ctypes.byref(aq), ctypes.byref(ak), _stream_handle(stream)))
    return q, k


def make_qk_rope(inv_freq, D, *, positions=None, rot_dim=None, interleaved=False, q_heads,
                 k_heads=0, q_norm_weight=None, k_norm_weight=None, norm_eps=1e-6) -> MgqaQkRope:
    """Fill an MgqaQkRope: inv_freq fp32 [rot_dim / 2] (rot_dim defaults to D),
    positions int32 (prefill [B, Lq]; decode step [B]) or None, optional fp32
    [D] norm weights."""
    rot_dim = D if rot_dim is None else int(rot_dim)
    if inv_freq is None:
        raise ValueError("inv_freq is required")
    _dev(inv_freq, "inv_freq", torch.float32)
    if not inv_freq.is_contiguous() or inv_freq.numel() != rot_dim // 2:
        raise ValueError(f"inv_freq must be a contiguous fp32 tensor of {rot_dim // 2} values")
    r = MgqaQkRope()
    r.inv_freq = inv_freq.data_ptr()
    if positions is not None:
        _dev(positions, "positions", torch.int32)
        if not positions.is_contiguous():
            raise ValueError("positions must be contiguous")
        r.positions = positions.data_ptr()
    r.rot_dim, r.interleaved = rot_dim, int(bool(interleaved))
    r.q_heads, r.k_heads = int(q_heads), int(k_heads)
    for name, t in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
        if t is not None:
            _dev(t, name, torch.float32)
            if not t.is_contiguous() or t.numel() != D:
                raise ValueError(f"{name} must be a contiguous fp32 tensor of {D} values")
            setattr(r, name, t.data_ptr())
    r.norm_eps = float(norm_eps)
    return r


def masked_gqa_attn_prefill_rope(q, k, v, out=None, *, inv_freq, positions=None, rot_dim=None,
                                 interleaved=False, q_heads=None, q_norm_weight=None,
                                 norm_eps=1e-6, scale=None, mask_bits=None, kv_len=None,
                                 seg_q=None, seg_k=None, lse=None, dev_error=None, causal=False,
                                 stream=None):
    """masked_gqa_attn_prefill with the rotary embedding (and optional RMS
    norm) applied to q inside the kernel; k must already be rotated. Returns out."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k, v, out, scale=scale, mask_bits=mask_bits, kv_len=kv_len, seg_q=seg_q,
                  seg_k=seg_k, lse=lse, dev_error=dev_error, causal=causal)
    if positions is not None and tuple(positions.shape) != (q.shape[0], q.shape[2]):
        raise ValueError("positions must be int32 [B, Lq]")
    r = make_qk_rope(inv_freq, q.shape[3], positions=positions, rot_dim=rot_dim,
                     interleaved=interleaved, q_heads=q.shape[1] if q_heads is None else q_heads,
                     q_norm_weight=q_norm_weight, norm_eps=norm_eps)
    _check(lib().masked_gqa_attn_prefill_rope(ctypes.byref(a), ctypes.byref(r),
                                              _stream_handle(stream)))
    return out


def masked_gqa_attn_decode_append_rope(q, k_cache, v_cache, k_new, v_new, kv_len, out=None, *,
                                       workspace: Optional[torch.Tensor] = None, inv_freq=None,
                                       positions=None,
                                       rot_dim=None, interleaved=False, q_heads=None,
                                       k_heads=None, q_norm_weight=None, k_norm_weight=None,
                                       norm_eps=1e-6, kv_len_out=None, scale=None, lse=None,
                                       dev_error=None, stream=None):
    """masked_gqa_attn_decode_append with the rotary embedding (and optional
    RMS norms) applied inside the kernel to q and to the new key row, at the
    new token's position (positions int32 [B], default kv_len); the cache
    receives the rotated key row. Returns out."""
    if out is None:
        out = torch.empty_like(q)
    a = make_args(q, k_cache, v_cache, out, scale=scale, kv_len=kv_len, lse=lse,
                  dev_error=dev_error)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _dev(t, name, q.dtype)
        if t.dim() != 4 or t.shape[2] != 1 or t.stride(3) != 1:
            raise ValueError(f"{name} must be [B, Hkv, 1, D] with a unit-stride head dim")
    if positions is not None and tuple(positions.shape) != (q.shape[0],):
        raise ValueError("positions must be int32 [B]")
    r = make_qk_rope(inv_freq, q.shape[3], positions=positions, rot_dim=rot_dim,
                     interleaved=interleaved, q_heads=q.shape[1] if q_heads is None else q_heads,
                     k_heads=k_cache.shape[1] if k_heads is None else k_heads,
                     q_norm_weight=q_norm_weight, k_norm_weight=k_norm_weight, norm_eps=norm_eps)
    ks = (ctypes.c_int64 * 2)(k_new.stride(0), k_new.stride(1))
    vs = (ctypes.c_int64 * 2)(v_new.stride(0), v_new.stride(1))
    wp, wn = _workspace(workspace)
    _check(lib().masked_gqa_attn_decode_append_rope(
        ctypes.byref(a), k_new.data_ptr(), v_new.data_ptr(), ks, vs,
        _ptr(_dev(kv_len_out, "kv_len_out", torch.int32)), ctypes.byref(r), wp, wn,
        _stream_handle(stream)))
    return out
