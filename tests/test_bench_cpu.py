"""Host-side pieces of the benchmark and the workload generators, checked
without a GPU: the algorithmic work each metric divides by, the seeded
inputs, the peak fallback and the profile lookup that feeds `traffic`."""
import hashlib
import importlib.util
import os

import pytest
import torch

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_padded_cfg_flops_closed_form():
    # rows of 1024 and 384 valid keys, every query row attends to all of them:
    # 4 * D * Hq * Lq * (1024 + 384)
    wl = W.padded_cfg(variant="bits")
    assert wl.flops() == 4.0 * 128 * 16 * 1024 * (1024 + 384)
    # 384 = 3 x 128: the non-empty 128 x 128 tiles hold exactly the allowed pairs
    assert wl.nonempty_tile_flops() == wl.flops()
    assert W.padded_cfg(variant="kvlen").flops() == wl.flops()


def test_packed_guidance_flops_closed_form():
    wl = W.packed_guidance()
    assert wl.flops() == 4.0 * 128 * 16 * (1024 * 1024 + 384 * 384)


def test_seeded_inputs_are_reproducible():
    a, b = W.padded_cfg(variant="bits"), W.padded_cfg(variant="bits")
    for n in ("q", "k", "v", "mask_bits"):
        assert torch.equal(getattr(a, n), getattr(b, n))
    c = W.padded_cfg(seed=7, variant="bits")
    assert not torch.equal(a.q, c.q)


def test_decode_needed_bytes_counts_filled_rows_only(bench):
    wl = W.static_cache_decode(variant="span")
    B, Hq, Hkv, Lq, Lk, D = wl.shape
    filled = int(wl.kv_len.sum())
    expect = filled * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2
    assert bench.decode_needed_bytes(wl) == expect
    full = W.static_cache_decode(variant="full")
    # the bitmask form also reads one bit per cache slot
    assert bench.decode_needed_bytes(full) == expect + B * (Lk // 32) * 4


def test_peak_fallback_when_not_measured(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d, kind = bench.peaks()
    assert kind == "fallback"
    assert d["hbm_gbs"] == 6800.0 and d["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"gpu": {"hbm_gbs": 7000.5, "bf16_tflops": 1888}}')
    d, kind = bench.peaks()
    assert kind == "measured"
    assert bench.peak_value(d, "hbm_gbs") == 7000.5
    assert bench.peak_value(d, "bf16_tflops") == 1888.0


def test_traffic_only_for_the_profiled_source(bench, tmp_path, monkeypatch):
    src_dir = tmp_path / "masked_gqa_attention_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "k.md").write_text(
        f"notes\n\ntraffic: 123456 source-sha256: {sha} k.cu\n"
        f"traffic: 777 source-sha256: {sha} k.cu other_workload\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("k.cu") == 123456.0
    assert bench.traffic_from_profiles("k.cu", "other_workload") == 777.0
    assert bench.traffic_from_profiles("k.cu", "missing_workload") is None
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.traffic_from_profiles("k.cu") is None
    assert bench.traffic_from_profiles("missing.cu") is None


def test_committed_profiles_name_their_sources():
    # every traffic line names a kernel file that exists and a 16-hex hash
    lines = []
    for f in os.listdir(os.path.join(ROOT, "profiles")):
        for line in open(os.path.join(ROOT, "profiles", f)):
            if line.startswith("traffic:"):
                lines.append(line.split())
    assert lines, "no traffic line in profiles/"
    for parts in lines:
        assert float(parts[1]) > 0
        assert parts[2] == "source-sha256:" and len(parts[3]) == 16
        int(parts[3], 16)
        assert os.path.exists(os.path.join(ROOT, "masked_gqa_attention_gb300", "csrc", parts[4]))


# ---- the input recipe: the structure every parity and invariance test relies on

def test_padded_cfg_mask_encodes_the_two_row_lengths():
    wl = W.padded_cfg(variant="bits")
    a = W.unpack_bits(wl.mask_bits, 1024)          # [B, Lq, Lk] bool
    assert a.shape == (2, 1024, 1024)
    assert bool(a[0].all())
    assert bool(a[1, :, :384].all()) and not bool(a[1, :, 384:].any())
    kv = W.padded_cfg(variant="kvlen")
    assert kv.kv_len.tolist() == [1024, 384]
    assert torch.equal(kv.allowed(), wl.allowed())


def test_static_cache_garbage_past_the_filled_length():
    wl = W.static_cache_decode(variant="span")
    filled = wl.kv_len.tolist()
    assert all(256 <= f <= 3100 for f in filled)
    for b, f in enumerate(filled):
        tail_k, tail_v = wl.k[b, :, f:].float(), wl.v[b, :, f:].float()
        # large finite values: if masked slots leaked into a result, it would show
        assert bool(torch.isfinite(tail_k).all()) and float(tail_k.abs().max()) > 1e3
        assert float(tail_v.abs().max()) > 1e3 and float(tail_v.abs().max()) <= 1e4
        assert float(wl.k[b, :, :f].float().abs().max()) < 10.0
    full = W.static_cache_decode(variant="full")
    assert torch.equal(full.allowed(), wl.allowed())
    assert torch.equal(full.k, wl.k) and torch.equal(full.v, wl.v)


def test_dit_segments_cut_rows_off_the_tile_grid():
    seg = W.dit_segments(1005, 32, 4096)
    counts = [int(seg[b].max()) + 1 for b in range(32)]
    assert min(counts) >= 1 and max(counts) <= 6 and len(set(counts)) > 1
    # ids are non-decreasing along a row (contiguous blocks)
    assert bool((seg[:, 1:] >= seg[:, :-1]).all())
    cuts = [c for b in range(32) for c in (torch.nonzero(seg[b, 1:] != seg[b, :-1]).flatten() + 1).tolist()]
    assert cuts and any(c % 128 != 0 for c in cuts)  # partial tiles occur


def test_cpu_oracle_block_whole_call(bench):
    wl = W.tiny_fp32()
    blk = bench.cpu_block(wl, "TFLOP/s", None, 0.01, sample="whole tiny call")
    assert blk["kind"] == "oracle" and blk["cores"] >= 1 and blk["value"] > 0
    assert blk["s_per_call"] > 0
    # TFLOP/s = allowed FLOPs / seconds per call
    assert abs(blk["value"] * 1e12 * blk["s_per_call"] - wl.flops()) < 1e-6 * wl.flops()


def test_cpu_oracle_block_row_sample_counts_the_sampled_rows(bench):
    wl = W.random_case(3, 4, 4, 2, 200, 200, 64, dtype=torch.bfloat16, mask="segment")
    f, secs, used = bench.cpu_oracle(wl, rows=[0, 2])
    sub = W.Workload("s", wl.q[[0, 2]], wl.k[[0, 2]], wl.v[[0, 2]], wl.scale,
                     seg_q=wl.seg_q[[0, 2]], seg_k=wl.seg_k[[0, 2]])
    assert f == sub.flops() and secs > 0 and used >= 1
    blk = bench.cpu_block(wl, "TFLOP/s", None, 0.01, rows=[0, 2], sample="rows 0, 2")
    # seconds per call extrapolate the sample to all 4 rows
    assert blk["s_per_call"] > 0


def test_cpu_oracle_block_bytes_for_decode(bench):
    wl = W.static_cache_decode(variant="span", B=2, capacity=512, lo=100, hi=400)
    nb = bench.decode_needed_bytes(wl)
    blk = bench.cpu_block(wl, "GB/s", nb, 0.01, sample="whole decode call")
    assert blk["unit"] == "GB/s" and abs(blk["value"] * 1e9 * blk["s_per_call"] - nb) < 1e-6 * nb


def test_fp32_alu_peak_from_unit_counts(bench):
    assert abs(bench.fp32_alu_peak_tflops() - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
