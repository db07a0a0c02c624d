"""Seeded synthetic inputs shaped like the engine pages' attention workloads.

This module draws random numbers and lays out masks; it holds none of the
attention arithmetic. Both the CUDA library's tests/benchmark and the fp64
oracle take their inputs from here, so the two sides see identical bytes.

Shapes follow the pages:
  * OmniVoice page, "Upstream-identical practice" and "Memory & speed":
    a bidirectional Qwen3 decoder (16 query heads, 8 KV heads, head_dim 128)
    run on a classifier-free-guidance batch of two rows, the unconditional
    row padded to the conditional length; or both packed into one row under
    a block-diagonal mask (packed_guidance).
  * VoxCPM page, "Upstream-identical practice" and "Memory & speed": one-token
    decode over a static 8192-slot KV cache whose slots past the filled length
    are masked (attention_span), and a bidirectional local DiT.

Values are ``torch.randn`` in fp32 from ``torch.Generator('cpu')`` seeded per
workload, then cast to the workload dtype. Masks are given as
  * ``mask_bits``: uint32 words [B, Lq, ceil(Lk/32)], bit j%32 of word j//32
    set when key j may be attended (least-significant bit first);
  * ``kv_len``: int32 [B], keys j < kv_len[b] valid;
  * ``seg_q`` / ``seg_k``: int32 [B, Lq] / [B, Lk] segment ids, attention only
    within equal non-negative ids.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


def pack_bool_mask(mask: torch.Tensor) -> torch.Tensor:
    """Pack a boolean [B, Lq, Lk] mask into uint32 words (returned as int32).

    Bit j % 32 of word j // 32 holds mask[..., j]; bits past Lk are zero.
    """
    mask = mask.to(torch.bool).cpu()
    B, Lq, Lk = mask.shape
    W = (Lk + 31) // 32
    padded = torch.zeros((B, Lq, W * 32), dtype=torch.bool)
    padded[:, :, :Lk] = mask
    m = padded.view(B, Lq, W, 32).to(torch.int64)
    weights = (torch.ones(32, dtype=torch.int64) << torch.arange(32, dtype=torch.int64))
    words = (m * weights).sum(-1)  # < 2**32, exact in int64
    words = torch.where(words >= 2**31, words - 2**32, words)
    return words.to(torch.int32).contiguous()


def unpack_bits(words: torch.Tensor, Lk: int) -> torch.Tensor:
    """Inverse of :func:`pack_bool_mask` (for tests and input checks)."""
    w = words.cpu().to(torch.int64) & 0xFFFFFFFF
    bits = (w.unsqueeze(-1) >> torch.arange(32, dtype=torch.int64)) & 1
    return bits.reshape(*w.shape[:-1], -1)[..., :Lk].to(torch.bool)


@dataclass
class Workload:
    """One attention call's inputs (CPU tensors) and its description."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    scale: float
    mask_bits: Optional[torch.Tensor] = None
    kv_len: Optional[torch.Tensor] = None
    seg_q: Optional[torch.Tensor] = None
    seg_k: Optional[torch.Tensor] = None
    causal: bool = False
    seed: int = 0
    info: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, Hq, Lq, D = self.q.shape
        _, Hkv, Lk, _ = self.k.shape
        return B, Hq, Hkv, Lq, Lk, D

    def allowed(self) -> torch.Tensor:
        """Boolean [B, Lq, Lk] of allowed (query, key) pairs (AND of the forms)."""
        B, Hq, Hkv, Lq, Lk, D = self.shape
        a = torch.ones((B, Lq, Lk), dtype=torch.bool)
        if self.mask_bits is not None:
            a &= unpack_bits(self.mask_bits, Lk)
        if self.kv_len is not None:
            a &= (torch.arange(Lk)[None, None, :] < self.kv_len.cpu()[:, None, None].to(torch.int64))
        if self.seg_q is not None:
            sq = self.seg_q.cpu()[:, :, None]
            sk = self.seg_k.cpu()[:, None, :]
            a &= (sq == sk) & (sq >= 0)
        if self.causal:
            i = torch.arange(Lq)[:, None]
            j = torch.arange(Lk)[None, :]
            a &= (j <= i + (Lk - Lq))[None]
        return a

    def masks(self) -> dict:
        d = dict(mask_bits=self.mask_bits, kv_len=self.kv_len,
                 seg_q=self.seg_q, seg_k=self.seg_k)
        if self.causal:
            d["causal"] = True
        return d

    def allowed_pairs(self) -> int:
        return int(self.allowed().sum())

    def flops(self) -> float:
        """Algorithmic FLOPs: 4*D per allowed (query, key) pair per query head."""
        B, Hq, Hkv, Lq, Lk, D = self.shape
        return 4.0 * D * Hq * self.allowed_pairs()

    def nonempty_tile_flops(self, tile: int = 128) -> float:
        """4*D*tile*tile per query head per non-empty tile x tile block."""
        B, Hq, Hkv, Lq, Lk, D = self.shape
        a = self.allowed()
        nq, nk = -(-Lq // tile), -(-Lk // tile)
        pad = torch.zeros((B, nq * tile, nk * tile), dtype=torch.bool)
        pad[:, :Lq, :Lk] = a
        blocks = pad.view(B, nq, tile, nk, tile).any(dim=4).any(dim=2)
        return 4.0 * D * Hq * tile * tile * float(blocks.sum())


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn(g, shape, dtype):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype).contiguous()


def random_qkv(seed, B, Hq, Hkv, Lq, Lk, D, dtype):
    g = _gen(seed)
    q = _randn(g, (B, Hq, Lq, D), dtype)
    k = _randn(g, (B, Hkv, Lk, D), dtype)
    v = _randn(g, (B, Hkv, Lk, D), dtype)
    return g, q, k, v


# --- the five named workloads ---------------------------------------------

def tiny_fp32(seed: int = 1001) -> Workload:
    """Tiny bidirectional masked GQA, fp32: B=2 (cond/uncond), Hq=4, Hkv=2,
    D=64, L=128, scale 1/8; row 0 attends to every key, row 1 only to the last
    48 keys (80..127) for every query."""
    B, Hq, Hkv, L, D = 2, 4, 2, 128, 64
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, L, L, D, torch.float32)
    mask = torch.ones((B, L, L), dtype=torch.bool)
    mask[1, :, :80] = False
    return Workload("tiny_fp32", q, k, v, 1.0 / 8.0, mask_bits=pack_bool_mask(mask),
                    seed=seed, info=dict(dtype="fp32"))


def padded_cfg(seed: int = 1002, variant: str = "bits") -> Workload:
    """OmniVoice-shaped padded CFG prefill: B=2, Hq=16, Hkv=8, D=128, L=1024,
    bf16; row 0 all 1024 keys valid, row 1 (unconditional) only keys 0..383;
    key-padding mask for every query row. variant "bits" gives the 4D mask as
    packed bits, "kvlen" the same mask as per-row key lengths."""
    B, Hq, Hkv, L, D = 2, 16, 8, 1024, 128
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, L, L, D, torch.bfloat16)
    lens = torch.tensor([1024, 384], dtype=torch.int32)
    w = Workload(f"padded_cfg_{variant}", q, k, v, 1.0 / math.sqrt(D), seed=seed,
                 info=dict(dtype="bf16", calls=32))
    if variant == "bits":
        mask = torch.arange(L)[None, None, :] < lens[:, None, None].to(torch.int64)
        w.mask_bits = pack_bool_mask(mask.expand(B, L, L))
    elif variant == "kvlen":
        w.kv_len = lens
    else:
        raise ValueError(variant)
    return w


def packed_guidance(seed: int = 1003) -> Workload:
    """Packed-guidance block-diagonal prefill: one row of 1024 + 384 = 1408
    positions, Hq=16, Hkv=8, D=128, bf16; segment 0 for positions 0..1023,
    segment 1 for 1024..1407."""
    B, Hq, Hkv, L, D = 1, 16, 8, 1408, 128
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, L, L, D, torch.bfloat16)
    seg = torch.zeros((B, L), dtype=torch.int32)
    seg[:, 1024:] = 1
    return Workload("packed_guidance", q, k, v, 1.0 / math.sqrt(D), seg_q=seg,
                    seg_k=seg.clone(), seed=seed,
                    info=dict(dtype="bf16", segments=[(0, 1024), (1024, 1408)]))


def static_cache_decode(seed: int = 1004, variant: str = "span",
                        B: int = 8, Hq: int = 16, Hkv: int = 2, D: int = 64,
                        capacity: int = 8192, lo: int = 256, hi: int = 3100,
                        dtype=torch.bfloat16) -> Workload:
    """Static-cache decode: B requests, one query token each, Hq=16, Hkv=2,
    D=64, bf16, 8192 cache slots per request; filled lengths uniform in
    [256, 3100] from the seed; slots past the filled length hold uniform
    values in [-1e4, 1e4]. variant "full" masks the whole 8192-slot cache with
    packed bits; variant "span" passes the filled lengths."""
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, 1, capacity, D, dtype)
    filled = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    for b in range(B):
        n = capacity - int(filled[b])
        gk = (torch.rand((Hkv, n, D), generator=g) * 2e4 - 1e4).to(dtype)
        gv = (torch.rand((Hkv, n, D), generator=g) * 2e4 - 1e4).to(dtype)
        k[b, :, int(filled[b]):, :] = gk
        v[b, :, int(filled[b]):, :] = gv
    w = Workload(f"static_cache_decode_{variant}", q, k, v, 1.0 / math.sqrt(D),
                 seed=seed, info=dict(dtype=str(dtype).replace("torch.", ""),
                                      filled=filled.tolist(), capacity=capacity))
    if variant == "full":
        mask = torch.arange(capacity)[None, None, :] < filled[:, None, None]
        w.mask_bits = pack_bool_mask(mask)
    elif variant == "span":
        w.kv_len = filled.to(torch.int32)
    else:
        raise ValueError(variant)
    return w


def dit_segments(seed: int, B: int, L: int) -> torch.Tensor:
    """Per-row segment ids: n ~ U{1..6} segments, n-1 distinct cut points drawn
    uniformly from 1..L-1 and sorted."""
    g = _gen(seed + 7919)
    seg = torch.zeros((B, L), dtype=torch.int32)
    for b in range(B):
        n = int(torch.randint(1, 7, (1,), generator=g))
        cuts = torch.randperm(L - 1, generator=g)[: n - 1] + 1
        cuts, _ = torch.sort(cuts)
        for c in cuts.tolist():
            seg[b, c:] += 1
    return seg


def dit_batch(seed: int = 1005, B: int = 32, L: int = 4096) -> Workload:
    """Large bidirectional DiT-style batch: 32 rows, Hq=16, Hkv=4, D=128,
    L=4096, bf16; each row split into 1..6 block-diagonal segments at cut
    points drawn from the seed (not tile-aligned)."""
    Hq, Hkv, D = 16, 4, 128
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, L, L, D, torch.bfloat16)
    seg = dit_segments(seed, B, L)
    return Workload("dit_batch", q, k, v, 1.0 / math.sqrt(D), seg_q=seg, seg_k=seg.clone(),
                    seed=seed, info=dict(dtype="bf16", calls=20))


def random_case(seed: int, B, Hq, Hkv, Lq, Lk, D, dtype=torch.bfloat16,
                mask: str = "bits", density: float = 0.7) -> Workload:
    """A generic seeded case for parity tests. mask is one of "none", "bits"
    (random key-padding and random per-element holes), "kvlen", "segment",
    "bits+kvlen", "causal"."""
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, Lq, Lk, D, dtype)
    w = Workload(f"random_{mask}", q, k, v, 1.0 / math.sqrt(D), seed=seed,
                 info=dict(dtype=str(dtype).replace("torch.", "")))
    if "bits" in mask:
        m = torch.rand((B, Lq, Lk), generator=g) < density
        # also make whole 128-key blocks fully on / fully off for some rows
        for b in range(B):
            lens = int(torch.randint(0, Lk + 1, (1,), generator=g))
            if b % 2 == 1:
                m[b, :, lens:] = False
            if b % 3 == 0:
                m[b, :, : min(Lk, 128)] = True
        w.mask_bits = pack_bool_mask(m)
    if "kvlen" in mask:
        w.kv_len = torch.randint(0, Lk + 1, (B,), generator=g, dtype=torch.int32)
        w.kv_len[0] = Lk
    if mask == "segment":
        seg = torch.zeros((B, max(Lq, Lk)), dtype=torch.int32)
        for b in range(B):
            n = int(torch.randint(1, 5, (1,), generator=g))
            L = max(Lq, Lk)
            cuts = torch.sort(torch.randperm(max(L - 1, 1), generator=g)[: n - 1] + 1)[0]
            for c in cuts.tolist():
                seg[b, c:] += 1
            if b % 2 == 1:  # padded head and tail positions that attend nowhere
                seg[b, L - L // 8:] = -1
                seg[b, : max(1, L // 16)] = -1
        w.seg_q = seg[:, :Lq].contiguous()
        w.seg_k = seg[:, :Lk].contiguous()
    if mask == "causal":
        w.causal = True
    if mask not in ("none", "bits", "kvlen", "segment", "bits+kvlen", "causal"):
        raise ValueError(mask)
    return w


def growing_scores(seed: int, B, Hq, Hkv, L, D, dtype=torch.bfloat16, mask: str = "none",
                   growth: float = 2.5, tile: int = 128) -> Workload:
    """Inputs whose row maxima climb from key tile to key tile: the keys of
    tile t are N(0,1) values times (1 + growth * t), so with q ~ N(0,1) and
    scale 1/sqrt(D) a row's largest score grows by about 2.6 * growth nats
    (well over 8 powers of two for growth 2.5) at every tile boundary. Real
    attention logits span that range; N(0,1) inputs never do. Such a softmax
    is peaked, so an output row is close to one value row; V is N(0,1) / 4 so
    that the outputs stay within the magnitude the absolute bf16 bound is set
    for (rows of N(0,1) averages). mask as in :func:`random_case` ("none",
    "bits", "segment")."""
    w = random_case(seed, B, Hq, Hkv, L, L, D, dtype=dtype, mask=mask)
    f = 1.0 + growth * (torch.arange(L) // tile).to(torch.float32)
    w.k = (w.k.to(torch.float32) * f[None, None, :, None]).to(dtype).contiguous()
    w.v = (w.v.to(torch.float32) * 0.25).to(dtype).contiguous()
    w.name = f"growing_scores_{mask}"
    w.info["growth"] = growth
    return w


def late_spike(seed: int, B, Hq, Hkv, L, D, dtype=torch.bfloat16, first: int = 127,
               spike: float = 6.0) -> Workload:
    """Two segments per row, [0, first) and [first, L): the second starts one
    key before a tile edge (first = 127). That key is scaled near zero, so
    the second segment's rows see one low score in their first non-empty
    tile, then keys scaled by `spike` (scores far higher) in the next ones."""
    g, q, k, v = random_qkv(seed, B, Hq, Hkv, L, L, D, dtype)
    kf = k.to(torch.float32)
    kf[:, :, first] *= 0.01
    kf[:, :, (first // 128 + 1) * 128:] *= spike
    seg = torch.zeros((B, L), dtype=torch.int32)
    seg[:, first:] = 1
    return Workload("late_spike", q, kf.to(dtype).contiguous(), v, 1.0 / math.sqrt(D),
                    seg_q=seg, seg_k=seg.clone(), seed=seed,
                    info=dict(dtype=str(dtype).replace("torch.", ""), first=first, spike=spike))


CONFIGS = {
    1: tiny_fp32,
    2: padded_cfg,
    3: packed_guidance,
    4: static_cache_decode,
    5: dit_batch,
}
