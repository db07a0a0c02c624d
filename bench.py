#!/usr/bin/env python3
"""Benchmark of the masked GQA attention library on synthetic engine-shaped
workloads; prints ONE JSON line (rank 0).

Headline workload (one "step"): the largest single-GPU configuration, the
DiT-style bidirectional batch -- 32 rows x 4096 positions, 16 query heads, 4
KV heads, head_dim 128, bf16, each row cut into 1..6 block-diagonal segments
at seeded, tile-unaligned cut points -- called 20 times (10 Euler steps x the
classifier-free-guidance pair). The inputs (805 MB) are larger than L2, the
step is captured once in a CUDA graph and replayed.

Every other configuration is measured in the same run and reported under
"configs", each with its own roofline block, CPU-oracle baseline and clock
sample: the tiny fp32 case, the OmniVoice-shaped padded CFG prefill (32 calls
per step over 8 rotating input sets, 201 MB), the packed-guidance prefill,
the static-cache decode (8 requests, 8192-slot caches filled 256..3100, 16
rotating cache sets of 33.5 MB), and the rotary embedding of the padded-CFG q
and k.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the headline workload (the baseline arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "masked GQA prefill TFLOP/s & cache-decode GB/s, as % of GB300 roofline"
DIT_CALLS = 20          # 10 Euler steps x the CFG pair
CFG_CALLS = 32          # the 32 unmasking steps of the padded-CFG prefill
PREFILL_SETS = 8
DECODE_SETS = 16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(d, *keys):
    for k in keys:
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k])
        for sub in d.values():
            if isinstance(sub, dict) and k in sub and isinstance(sub[k], (int, float)):
                return float(sub[k])
    return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_secs: float) -> float:
    """Replicas: every rank processes the same units; the job rate is all
    ranks' units over the slowest rank's time."""
    return world * units_per_rank / max_secs


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def device_inputs(wl, dev):
    d = {}
    for n in ("q", "k", "v", "mask_bits", "kv_len", "seg_q", "seg_k"):
        t = getattr(wl, n)
        d[n] = None if t is None else t.to(dev)
    return d


def make_args(M, d, out, wl, lse=None):
    return M.make_args(d["q"], d["k"], d["v"], out, scale=wl.scale, mask_bits=d["mask_bits"],
                       kv_len=d["kv_len"], seg_q=d["seg_q"], seg_k=d["seg_k"], lse=lse)


def time_graph(step_fn, steps, warmup, stream, world):
    """Capture step_fn in a CUDA graph; time exactly `steps` replays."""
    with torch.cuda.stream(stream):
        for _ in range(2):
            step_fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step_fn()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3, g


# ---------------------------------------------------------------- workloads

def bench_prefill_graph(M, wl, dev, calls, nsets, steps, warmup, world):
    """Device-resident inputs, rotating sets, step = `calls` prefill calls."""
    import ctypes
    base = device_inputs(wl, dev)
    sets = []
    for s in range(nsets):
        d = {n: (t.clone() if t is not None else None) for n, t in base.items()}
        out = torch.empty_like(d["q"])
        sets.append((d, out, make_args(M, d, out, wl)))
    L = M.lib()
    stream = torch.cuda.Stream(device=dev)

    def step():
        h = stream.cuda_stream
        for c in range(calls):
            a = sets[c % nsets][2]
            st = L.masked_gqa_attn_prefill(ctypes.byref(a), h)
            if st != 0:
                raise RuntimeError(f"prefill failed: {L.mgqa_last_error_detail()}")

    secs, _ = time_graph(step, steps, warmup, stream, world)
    return secs, sets


def bench_rope(M, dev, reps=20, warmup=3, nsets=12):
    """Rotary embedding of the headline shapes' q [2,16,1024,128] and
    k [2,8,1024,128] (bf16, full rotary dim, positions = row index); one call =
    q and k of one of `nsets` rotating sets, rotated by one masked_gqa_rope_pair
    launch (and, for comparison, by two masked_gqa_rope calls). One pass over
    the sets is captured in a CUDA graph (no host launch cost in the timed
    region) and replayed. Returns (seconds per call with the pair launch,
    seconds per call with two calls, algorithmic bytes per call: every rotated
    element read and written, plus the frequency table)."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(1006)
    sets = [(torch.randn(2, 16, 1024, 128, generator=g).to(torch.bfloat16).to(dev),
             torch.randn(2, 8, 1024, 128, generator=g).to(torch.bfloat16).to(dev)) for _ in range(nsets)]
    f = (10000.0 ** (-torch.arange(0, 128, 2, dtype=torch.float64) / 128)).to(torch.float32).to(dev)

    def time_pass(pair):
        def one_pass():
            for q, k in sets:
                if pair:
                    M.masked_gqa_rope_pair(q, k, f)
                else:
                    M.masked_gqa_rope(q, f)
                    M.masked_gqa_rope(k, f)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            one_pass()  # warm-up and lazy set-up outside the capture
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_pass()
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / (reps * nsets)

    t_pair, t_two = time_pass(True), time_pass(False)
    q, k = sets[0]
    nbytes = 2 * (q.numel() + k.numel()) * q.element_size() + f.numel() * 4
    return t_pair, t_two, nbytes


def time_calls(fn, reps=20, warmup=3):
    """Capture fn (a sequence of launches on the current stream) in a CUDA
    graph; seconds per replay over `reps` replays."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def bench_fused_rope(M, dev, nsets=8):
    """The rotary embedding with the Qwen3-style q/k norm, fused into the
    attention against the standalone kernel followed by the plain call:
    (a) the padded-CFG prefill (q rotated in the kernel; k pre-rotated), (b)
    the static-cache decode step with its append. Seconds per call."""
    f128 = (10000.0 ** (-torch.arange(0, 128, 2, dtype=torch.float64) / 128)).to(torch.float32).to(dev)
    f64 = (10000.0 ** (-torch.arange(0, 64, 2, dtype=torch.float64) / 64)).to(torch.float32).to(dev)
    g = torch.Generator().manual_seed(1007)
    w128 = (0.5 + torch.rand(128, generator=g)).to(dev)
    w64 = (0.5 + torch.rand(64, generator=g)).to(dev)
    wl = W.padded_cfg(variant="kvlen")
    sets = []
    for _ in range(nsets):
        d = device_inputs(wl, dev)
        sets.append((d, torch.empty_like(d["q"])))

    def prefill_fused():
        for d, out in sets:
            M.masked_gqa_attn_prefill_rope(d["q"], d["k"], d["v"], out, inv_freq=f128,
                                           q_norm_weight=w128, scale=wl.scale, kv_len=d["kv_len"])

    def prefill_unfused():
        for d, out in sets:
            M.masked_gqa_rope(d["q"], f128, norm_weight=w128)
            M.masked_gqa_attn_prefill(d["q"], d["k"], d["v"], out, scale=wl.scale, kv_len=d["kv_len"])

    tp_f = time_calls(prefill_fused) / nsets
    tp_u = time_calls(prefill_unfused) / nsets
    del sets
    wd = W.static_cache_decode(variant="span")
    B, Hq, Hkv, _, Lk, D = wd.shape
    dsets = []
    for _ in range(DECODE_SETS):
        d = device_inputs(wd, dev)
        kn = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).to(dev)
        vn = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).to(dev)
        dsets.append((d, kn, vn, torch.empty_like(d["kv_len"]), torch.empty_like(d["q"])))
    pos = [ds[0]["kv_len"][:, None].contiguous() for ds in dsets]

    def step_fused():
        for d, kn, vn, lo, out in dsets:
            M.masked_gqa_attn_decode_append_rope(d["q"], d["k"], d["v"], kn, vn, d["kv_len"], out,
                                                 inv_freq=f64, q_norm_weight=w64,
                                                 k_norm_weight=w64, kv_len_out=lo, scale=wd.scale)

    def step_unfused():
        for (d, kn, vn, lo, out), p in zip(dsets, pos):
            M.masked_gqa_rope_pair(d["q"], kn, f64, positions=p, q_norm_weight=w64, k_norm_weight=w64)
            M.masked_gqa_attn_decode_append(d["q"], d["k"], d["v"], kn, vn, d["kv_len"], out,
                                            kv_len_out=lo, scale=wd.scale)

    td_f = time_calls(step_fused) / DECODE_SETS
    td_u = time_calls(step_unfused) / DECODE_SETS
    return tp_f, tp_u, td_f, td_u


def decode_needed_bytes(wl):
    B, Hq, Hkv, Lq, Lk, D = wl.shape
    es = wl.k.element_size()
    filled = sum(int(x) for x in wl.allowed()[:, 0, :].sum(-1))
    kv = filled * Hkv * D * 2 * es
    qo = 2 * B * Hq * D * es
    mask = 0 if wl.mask_bits is None else B * ((Lk + 31) // 32) * 4
    return kv + qo + mask


def bench_decode(M, wl, dev, steps, warmup, world, nsets=DECODE_SETS, calls=16):
    import ctypes
    base = device_inputs(wl, dev)
    sets = []
    for s in range(nsets):
        d = {n: (t.clone() if t is not None else None) for n, t in base.items()}
        out = torch.empty_like(d["q"])
        a = make_args(M, d, out, wl)
        masks = {n: d[n] for n in ("mask_bits", "kv_len", "seg_q", "seg_k")}
        sets.append((d, out, a))
    L = M.lib()
    stream = torch.cuda.Stream(device=dev)

    def step():
        for c in range(calls):
            d, out, a = sets[c % nsets]
            st = L.masked_gqa_attn_decode(ctypes.byref(a), None, 0, stream.cuda_stream)
            if st != 0:
                raise RuntimeError(L.mgqa_last_error_detail())

    secs, _ = time_graph(step, steps, warmup, stream, world)
    return secs / (steps * calls)


def bench_decode_e2e(M, wl, dev, steps, warmup, world):
    """Per step: H2D of the new query and lengths, one decode call, D2H of the
    output (the cache stays resident, as a static KV cache does). Steps run one
    after another, as a token loop's do. The query and the lengths travel in
    one pinned buffer (one copy), and the step is captured once in a CUDA
    graph, as the pages' decode loop is."""
    import ctypes
    d = device_inputs(wl, dev)
    qb = wl.q.numel() * wl.q.element_size()
    nl = wl.kv_len.numel() if wl.kv_len is not None else 0
    # [q bytes | kv_len bytes] on the host (pinned) and on the device
    hbuf = torch.empty(qb + 4 * nl, dtype=torch.uint8).pin_memory()
    hbuf[:qb].copy_(wl.q.contiguous().view(-1).view(torch.uint8))
    if nl:
        hbuf[qb:].copy_(wl.kv_len.contiguous().view(-1).view(torch.uint8))
    dbuf = torch.empty(qb + 4 * nl, dtype=torch.uint8, device=dev)
    d["q"] = dbuf[:qb].view(wl.q.dtype).view(wl.q.shape)
    if nl:
        d["kv_len"] = dbuf[qb:].view(torch.int32).view(wl.kv_len.shape)
    out = torch.empty_like(d["q"])
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    a = make_args(M, d, out, wl)
    L = M.lib()
    stream = torch.cuda.Stream(device=dev)

    def step():
        dbuf.copy_(hbuf, non_blocking=True)
        st = L.masked_gqa_attn_decode(ctypes.byref(a), None, 0, stream.cuda_stream)
        if st != 0:
            raise RuntimeError(L.mgqa_last_error_detail())
        oh.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps, qb + 4 * nl, oh.numel() * oh.element_size()


def traffic_from_profiles(kernel_file: str, workload: str = None):
    """DRAM bytes per launch recorded by an ncu capture of the current kernel
    source (profiles/*.md line 'traffic: <bytes> source-sha256: <hex> <file>
    [<workload>]'), or None."""
    import glob
    import hashlib
    src = os.path.join(ROOT, "masked_gqa_attention_gb300", "csrc", kernel_file)
    if not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for p in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(p):
            parts = line.split()
            if (len(parts) >= 5 and parts[0] == "traffic:" and parts[2] == "source-sha256:"
                    and parts[3] == sha and parts[4] == kernel_file
                    and (workload is None or (len(parts) > 5 and parts[5] == workload))):
                try:
                    return float(parts[1])
                except ValueError:
                    pass
    return None


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle(wl, rows=None, heads=None):
    """Time one oracle call on the rows / leading query heads given (all by
    default); returns (allowed FLOPs of the sample, seconds, threads used)."""
    import oracle
    oracle.build()
    q, k, v = wl.q, wl.k, wl.v
    masks = wl.masks()
    if rows is not None:
        q, k, v = q[rows], k[rows], v[rows]
        masks = {n: (t[rows] if (t is not None and n != "causal") else t) for n, t in masks.items()}
    n_rep = wl.q.shape[1] // wl.k.shape[1]
    if heads is not None:
        hk = max(1, math.ceil(heads / n_rep))
        q, k, v = q[:, :heads], k[:, :hk], v[:, :hk]
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    t0 = time.perf_counter()
    _, _, used = oracle.attention(q, k, v, scale=wl.scale, **masks)
    secs = time.perf_counter() - t0
    B = wl.q.shape[0]
    frac = (len(rows) / B if rows is not None else 1.0) * ((heads or wl.q.shape[1]) / wl.q.shape[1])
    if rows is not None:  # allowed pairs of the sampled rows only
        sub = W.Workload("sample", wl.q[rows], wl.k[rows], wl.v[rows], wl.scale,
                         **{n: (t[rows] if t is not None else None) for n, t in
                            dict(mask_bits=wl.mask_bits, kv_len=wl.kv_len, seg_q=wl.seg_q,
                                 seg_k=wl.seg_k).items()})
        flops = sub.flops() * ((heads or wl.q.shape[1]) / wl.q.shape[1])
    else:
        flops = wl.flops() * frac
    return flops, secs, used


def cpu_block(wl, unit, work_of_call, min_secs, rows=None, heads=None, sample=""):
    """The oracle on the host cores, repeated for at least min_secs; value in
    `unit` per second (TFLOP/s from FLOPs, GB/s from bytes)."""
    tot_w, tot_s, reps, used = 0.0, 0.0, 0, 0
    while tot_s < min_secs and reps < 200:
        f, secs, used = cpu_oracle(wl, rows=rows, heads=heads)
        w = f if work_of_call is None else work_of_call * (
            (len(rows) / wl.q.shape[0]) if rows is not None else 1.0)
        tot_w += w
        tot_s += secs
        reps += 1
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    return {"value": tot_w / tot_s / scale, "unit": unit, "cores": used, "kind": "oracle",
            "sample": f"{reps} x {sample}, {tot_s:.1f} s",
            "s_per_call": tot_s / reps / ((len(rows) / wl.q.shape[0]) if rows is not None else 1.0)}


# ---------------------------------------------------------------- blocks

def prefill_roofline(wl, per_call, bf16, pk_kind, workload):
    f = wl.flops()
    return {"bound": "tensor", "achieved": f / per_call / 1e12, "peak": bf16, "unit": "TFLOP/s",
            "frac": f / per_call / 1e12 / bf16,
            "traffic": traffic_from_profiles("prefill_tc.cu", workload),
            "peak_kind": f"bf16 burst, {pk_kind}", "flops_per_launch": f,
            "nonempty_tile_TFLOP_s": wl.nonempty_tile_flops() / per_call / 1e12,
            "frac_nonempty_tiles": wl.nonempty_tile_flops() / per_call / 1e12 / bf16,
            "kernel": "prefill_tc"}


def fp32_alu_peak_tflops():
    """FP32 FMA peak of the CUDA cores: 152 SMs x 128 FP32 lanes x 2 FLOPs x
    2.07 GHz (the maximum SM clock)."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = W.dit_batch()
    rows, heads = [0], 4
    for _ in range(args.warmup):
        cpu_oracle(wl, rows=rows, heads=heads)
    tot_f, tot_s, used = 0.0, 0.0, 0
    for _ in range(args.steps):
        f, s, used = cpu_oracle(wl, rows=rows, heads=heads)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e12
    sample = (f"batch row 0, query heads 0..{heads - 1} of one DiT-batch prefill call "
              f"(4096 positions, head_dim 128, that row's segments) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "dit_batch (B=32, Hq=16, Hkv=4, D=128, L=4096; 1..6 segments per row)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def bench_dit_e2e(M, wl, dev, calls, steps, warmup, world):
    """Through the C ABI from pinned host buffers: every call of a step copies
    its q/k/v and segment ids in and its output back out. The calls are
    pipelined the way a throughput user would run them: two device input and
    output sets; call i+1's inputs go in on a copy stream and call i-1's output
    comes out on another while call i computes (events order each buffer's
    reuse), so the host link and the kernel overlap. (Spreading each copy over
    several copy streams measured no faster: the host link is the limit.)"""
    import ctypes
    host = {n: (getattr(wl, n).pin_memory() if getattr(wl, n) is not None else None)
            for n in ("q", "k", "v", "mask_bits", "kv_len", "seg_q", "seg_k")}
    sets = []
    for _ in range(2):
        d = {n: (torch.empty_like(t, device=dev) if t is not None else None) for n, t in host.items()}
        out = torch.empty_like(d["q"])
        sets.append({"d": d, "out": out, "args": make_args(M, d, out, wl),
                     "out_host": torch.empty_like(host["q"]).pin_memory()})
    L = M.lib()
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "run", "out")}
    h2d = calls * sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = calls * sets[0]["out_host"].numel() * sets[0]["out_host"].element_size()

    def step():
        for i in range(calls):
            b = i % 2
            st = sets[b]
            with torch.cuda.stream(s_in):  # inputs of call i, once call i-2 has read this set
                s_in.wait_event(ev["run"][b])
                for n, t in host.items():
                    if t is not None:
                        st["d"][n].copy_(t, non_blocking=True)
                ev["in"][b].record(s_in)
            s_run.wait_event(ev["in"][b])
            s_run.wait_event(ev["out"][b])  # call i-2's output has left this set
            rc = L.masked_gqa_attn_prefill(ctypes.byref(st["args"]), s_run.cuda_stream)
            if rc != 0:
                raise RuntimeError(L.mgqa_last_error_detail())
            ev["run"][b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["run"][b])
                st["out_host"].copy_(st["out"], non_blocking=True)
                ev["out"][b].record(s_out)

    main = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for s in (s_in, s_run, s_out):
        s.wait_event(e0)
    for _ in range(steps):
        step()
    for s in (s_in, s_run, s_out):
        main.wait_stream(s)
    e1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


def run_gpu(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import masked_gqa_attention_gb300 as M
    M.build_library()
    M.lib()
    pk, pk_kind = peaks()
    hbm = peak_value(pk, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    bf16 = peak_value(pk, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]

    if args.only is not None:  # profiling aid: one leg, raw timings
        if args.only == "decode":
            t = bench_decode(M, W.static_cache_decode(variant="span"), dev, args.steps,
                             args.warmup, world)
            print(json.dumps({"leg": "decode", "us_per_call": t * 1e6}))
            return 0
        maker, calls, nsets = {"prefill": (lambda: W.padded_cfg(variant="bits"), CFG_CALLS, PREFILL_SETS),
                               "prefill_kvlen": (lambda: W.padded_cfg(variant="kvlen"), CFG_CALLS,
                                                 PREFILL_SETS),
                               "packed": (W.packed_guidance, 32, PREFILL_SETS),
                               "tiny": (W.tiny_fp32, 32, 8),
                               "dit": (lambda: W.dit_batch(B=args.rows or 32), DIT_CALLS, 1)}[args.only]
        secs, _ = bench_prefill_graph(M, maker(), dev, calls, nsets, args.steps, args.warmup, world)
        print(json.dumps({"leg": args.only, "us_per_call": secs / (args.steps * calls) * 1e6}))
        return 0

    clocks = ClockSampler(local)
    cpu = rank == 0 and not args.no_cpu_baseline
    configs = {}

    # ---- headline: the DiT batch, 20 calls per step
    wl = W.dit_batch()
    clocks.start()
    secs, _ = bench_prefill_graph(M, wl, dev, DIT_CALLS, 1, args.steps, args.warmup, world)
    clk = clocks.stop()
    secs = max_over_ranks(secs, world)
    calls = args.steps * DIT_CALLS
    per_call = secs / calls
    value = whole_job_rate(calls * wl.flops(), world, secs) / 1e12
    roof = prefill_roofline(wl, per_call, bf16, pk_kind, "dit_batch")
    e2e_steps = 2
    e2e_secs, h2d, d2h = bench_dit_e2e(M, wl, dev, DIT_CALLS, e2e_steps, 1, world)
    e2e_secs = max_over_ranks(e2e_secs, world)
    e2e_value = whole_job_rate(e2e_steps * DIT_CALLS * wl.flops(), world, e2e_secs) / 1e12
    dit_cpu = None
    if cpu:
        dit_cpu = cpu_block(wl, "TFLOP/s", None, 2.0, rows=[0, 13], sample=(
            "batch rows 0 and 13 (all 16 heads, 4096 queries, their own segments) of one DiT "
            "call; s_per_call extrapolates to the 32 rows"))
    configs["dit_batch"] = {
        "workload": "B=32, Hq=16, Hkv=4, D=128, L=4096, bf16, 1..6 segments per row; 20 calls per step",
        "us_per_call": per_call * 1e6, "value": roof["achieved"], "unit": "TFLOP/s",
        "roofline": roof, "clocks": clk, "cpu_baseline": dit_cpu}
    del wl
    torch.cuda.empty_cache()

    # ---- padded CFG prefill (bits and kv_len forms), 32 calls per step
    for variant in ("bits", "kvlen"):
        wc = W.padded_cfg(variant=variant)
        clocks.start()
        so, _ = bench_prefill_graph(M, wc, dev, CFG_CALLS, PREFILL_SETS, 20, 3, world)
        ck = clocks.stop()
        pc = so / (20 * CFG_CALLS)
        blk = {"workload": f"B=2 CFG rows (keys 1024 / 384 valid), Hq=16, Hkv=8, D=128, L=1024, bf16, "
                           f"{'4D key-padding mask as packed bits' if variant == 'bits' else 'per-row key lengths'}; "
                           f"32 calls per step over {PREFILL_SETS} rotating sets (201 MB > L2)",
               "us_per_call": pc * 1e6, "unit": "TFLOP/s",
               "roofline": prefill_roofline(wc, pc, bf16, pk_kind, f"padded_cfg_{variant}"), "clocks": ck}
        blk["value"] = blk["roofline"]["achieved"]
        if cpu and variant == "bits":
            blk["cpu_baseline"] = cpu_block(wc, "TFLOP/s", None, 3.0,
                                            sample="whole padded-CFG prefill call (2 rows x 16 heads x 1024 queries)")
        configs[f"padded_cfg_{variant}"] = blk
        del wc

    # ---- packed guidance prefill
    wp = W.packed_guidance()
    clocks.start()
    so, _ = bench_prefill_graph(M, wp, dev, 32, PREFILL_SETS, 20, 3, world)
    ck = clocks.stop()
    pc = so / (20 * 32)
    configs["packed_guidance"] = {
        "workload": "1 row of 1024 + 384 positions, segments 0 / 1, Hq=16, Hkv=8, D=128, bf16; 32 calls "
                    f"per step over {PREFILL_SETS} rotating sets",
        "us_per_call": pc * 1e6, "unit": "TFLOP/s",
        "roofline": prefill_roofline(wp, pc, bf16, pk_kind, "packed_guidance"),
        "clocks": ck}
    configs["packed_guidance"]["value"] = configs["packed_guidance"]["roofline"]["achieved"]
    if cpu:
        configs["packed_guidance"]["cpu_baseline"] = cpu_block(
            wp, "TFLOP/s", None, 2.0, sample="whole packed-guidance prefill call (16 heads x 1408 queries)")

    # ---- tiny fp32 (CUDA cores)
    wt = W.tiny_fp32()
    clocks.start()
    so, _ = bench_prefill_graph(M, wt, dev, 32, 8, 20, 3, world)
    ck = clocks.stop()
    pc = so / (20 * 32)
    alu = fp32_alu_peak_tflops()
    configs["tiny_fp32"] = {
        "workload": "B=2, Hq=4, Hkv=2, D=64, L=128, fp32, key padding (row 1: last 48 keys); 32 calls per step",
        "us_per_call": pc * 1e6, "value": wt.flops() / pc / 1e12, "unit": "TFLOP/s",
        "roofline": {"bound": "alu", "achieved": wt.flops() / pc / 1e12, "peak": alu, "unit": "TFLOP/s",
                     "frac": wt.flops() / pc / 1e12 / alu, "traffic": None,
                     "peak_kind": "FP32 FMA: 152 SMs x 128 lanes x 2 x 2.07 GHz", "kernel": "prefill_simt"},
        "clocks": ck}
    if cpu:
        configs["tiny_fp32"]["cpu_baseline"] = cpu_block(wt, "TFLOP/s", None, 1.0,
                                                         sample="whole tiny fp32 call")

    # ---- static-cache decode: full-cache bitmask and filled-span forms
    for variant in ("span", "full"):
        wd = W.static_cache_decode(variant=variant)
        clocks.start()
        t = bench_decode(M, wd, dev, 30, 5, world)
        ck = clocks.stop()
        nb = decode_needed_bytes(wd)
        blk = {"workload": f"B=8, Hq=16, Hkv=2, D=64, bf16, 8192-slot caches filled 256..3100 "
                           f"({'per-row filled lengths' if variant == 'span' else 'full-cache bitmask'}); "
                           f"{DECODE_SETS} rotating cache sets (537 MB > L2)",
               "us_per_call": t * 1e6, "value": nb / t / 1e9, "unit": "GB/s",
               "roofline": {"bound": "hbm", "achieved": nb / t / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": nb / t / 1e9 / hbm,
                            "traffic": traffic_from_profiles("decode.cu", "static_cache_decode"),
                            "peak_kind": pk_kind, "bytes_per_launch": nb, "kernel": "decode"},
               "clocks": ck}
        if variant == "span":
            de2e, dh2d, dd2h = bench_decode_e2e(M, wd, dev, 200, 20, world)
            blk["e2e"] = {"value": nb / de2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": dh2d,
                          "d2h_bytes_per_step": dd2h}
            if cpu:
                blk["cpu_baseline"] = cpu_block(wd, "GB/s", nb, 1.0,
                                                sample="whole decode call (8 requests x 16 heads)")
        configs[f"static_cache_decode_{variant}"] = blk

    # ---- rotary embedding of the padded-CFG q and k
    clocks.start()
    t_rope, t_rope2, b_rope = bench_rope(M, dev)
    ck = clocks.stop()
    configs["rope_qk"] = {"workload": "rotary embedding of q [2,16,1024,128] and k [2,8,1024,128], "
                                      "bf16, 12 rotating sets (144 MB > L2); one pair launch per call",
                          "us_per_call": t_rope * 1e6, "two_calls_us": t_rope2 * 1e6,
                          "value": b_rope / t_rope / 1e9, "unit": "GB/s",
                          "roofline": {"bound": "hbm", "achieved": b_rope / t_rope / 1e9, "peak": hbm,
                                       "unit": "GB/s", "frac": b_rope / t_rope / 1e9 / hbm,
                                       "traffic": traffic_from_profiles("rope.cu"),
                                       "peak_kind": pk_kind, "bytes_per_launch": b_rope,
                                       "kernel": "rope"},
                          "clocks": ck}

    # ---- the rotary embedding (+ q/k RMS norm) fused into the attention calls
    clocks.start()
    tp_f, tp_u, td_f, td_u = bench_fused_rope(M, dev)
    ck = clocks.stop()
    wr = W.padded_cfg(variant="kvlen")
    configs["fused_rope"] = {
        "workload": "rotary embedding with the q/k RMS norm (fp32 table, half-split pairs, all heads) "
                    "inside the call: padded-CFG prefill (kv_len form; q rotated in the kernel, k "
                    "already rotated) and the static-cache decode step with its append (q and the new "
                    "key row rotated in the kernel), each against the standalone rotation (decode step: "
                    "q and the key row in one masked_gqa_rope_pair launch) + the plain call",
        "prefill_fused_us": tp_f * 1e6, "prefill_unfused_us": tp_u * 1e6,
        "prefill_fused_TFLOP_s": wr.flops() / tp_f / 1e12,
        "decode_step_fused_us": td_f * 1e6, "decode_step_unfused_us": td_u * 1e6,
        "value": tp_u / tp_f, "unit": "x (prefill: unfused time / fused time)",
        "roofline": {"bound": "tensor", "achieved": wr.flops() / tp_f / 1e12, "peak": bf16,
                     "unit": "TFLOP/s", "frac": wr.flops() / tp_f / 1e12 / bf16, "traffic": None,
                     "peak_kind": f"bf16 burst, {pk_kind}", "kernel": "prefill_tc (fused rotary)"},
        "clocks": ck}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "dit_batch: B=32 rows, Hq=16, Hkv=4, D=128, L=4096, bf16, 1..6 "
                               "block-diagonal segments per row at seeded cut points; 20 calls per step "
                               "(10 Euler steps x CFG pair)",
                   "l2": "inputs 805 MB > L2 (no rotation needed)",
                   "graph": "each step captured once in a CUDA graph", "parallelism": f"replicas x{world}"},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": calls,
        "roofline": roof,
        "configs": configs,
    }
    if dit_cpu is not None:
        line["cpu_baseline"] = {k: v for k, v in dit_cpu.items() if k != "s_per_call"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mgqa", choices=["mgqa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["prefill", "prefill_kvlen", "packed", "tiny", "dit", "decode"], default=None,
                    help="profiling aid: time only one workload (padded-CFG prefill, packed "
                         "guidance, DiT batch or the decode) and print its raw timing")
    ap.add_argument("--rows", type=int, default=None,
                    help="with --only dit: the first ROWS batch rows of the DiT workload (a "
                         "smaller capture of the same kernel)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
