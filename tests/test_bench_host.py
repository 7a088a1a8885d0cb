"""Host logic of the benchmark (no GPU): the algorithmic byte counts behind the roofline, the
guard that drops DRAM traffic recorded for another kernel source, and the peak lookup.

The byte counts are checked against per-workload closed forms written out independently of
``bench.algorithmic_bytes`` (the same numbers as the workload table of the design: inputs read
once, outputs written once, read too when accumulating).
"""
import json
import os

import numpy as np
import pytest

import bench
import workloads as W
import workloads.mgrouped as MW


def _closed_form(name):
    w = W.NAMED[name]()
    H, I, E, T = w.hidden, w.intermediate, w.num_experts, w.tokens_sum
    nonempty = int((np.asarray(w.counts) > 0).sum())
    if name == "balanced":      # BF16 in, FP32 dense out, overwrite
        return 2 * (H + I) * T + E * H * I * 4
    if name == "wide":          # BF16 in, BF16 dense out, accumulate: the non-empty experts read and write
        return 2 * (H + I) * T + 2 * nonempty * H * I * 2
    if name == "skewed":        # BF16 in, 128 discrete BF16 outputs, all written (zeros for empty experts)
        return 2 * (H + I) * T + E * H * I * 2
    if name == "fp8":           # e4m3 in + one FP32 scale per 128 tokens per row/column, BF16 out
        return (H + I) * T + (H + I) * (T // 128) * 4 + E * H * I * 2
    if name == "fp4":           # e2m1 (two per byte) + one UE8M0 byte per 32 tokens per row/column, BF16 out
        return (H + I) * T // 2 + (H + I) * (T // 32) + E * H * I * 2
    raise KeyError(name)


@pytest.mark.parametrize("name", ["balanced", "wide", "skewed", "fp8", "fp4"])
def test_algorithmic_bytes_match_closed_forms(name):
    assert bench.algorithmic_bytes(W.NAMED[name]()) == _closed_form(name)


def test_balanced_bytes_and_intensity_put_it_above_the_ridge():
    w = W.NAMED["balanced"]()
    intensity = w.flops / bench.algorithmic_bytes(w)
    ridge = 1946.0e12 / 6781.1e9
    assert 700 < intensity < 900 and intensity > ridge


def test_mgrouped_bytes_count_valid_rows_only():
    w = MW.MG_NAMED["mg_masked"]()
    rows, G = int(np.sum(w.counts)), w.num_groups
    # A's valid rows, every (non-empty) group's weight, D's valid rows; BF16 everywhere
    assert bench.mg_algorithmic_bytes(w) == rows * w.k * 2 + G * w.n * w.k * 2 + rows * w.n * 2
    wf = MW.MG_NAMED["mg_fp8_masked"]()
    expect = rows * wf.k + G * wf.n * wf.k + rows * wf.n * 2 + (rows + G * wf.n) * (wf.k // 128) * 4
    assert bench.mg_algorithmic_bytes(wf) == expect


def test_traffic_is_reported_only_for_the_kernel_it_was_measured_on(monkeypatch):
    rec = bench.traffic_record("balanced")
    path = os.path.join(bench.ROOT, "profiles", "traffic_balanced.json")
    with open(path) as f:
        d = json.load(f)
    if d["kernel_hash"] == bench.kernel_hash():
        assert rec == d["dram_bytes_per_launch"]
    else:
        assert rec is None
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.traffic_record("balanced") is None
    assert bench.traffic_record("no_such_workload") is None


def test_kernel_hash_follows_the_kernel_sources():
    h = bench.kernel_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert h == bench.kernel_hash()
    assert all(os.path.exists(os.path.join(bench.ROOT, f)) for f in bench.KERNEL_SOURCES)


def test_measured_peaks_come_from_the_driver_file_when_present():
    p = bench.measured_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured"
        assert p["bf16_tflops"] > 1000 and p["hbm_gbs"] > 1000
    else:
        assert p["source"] == "fallback"
