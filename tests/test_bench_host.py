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
    if name == "nvfp4":         # e2m1 (two per byte) + one UE4M3 byte per 16 tokens per row/column, BF16 out
        return (H + I) * T // 2 + (H + I) * (T // 16) + E * H * I * 2
    raise KeyError(name)


@pytest.mark.parametrize("name", ["balanced", "wide", "skewed", "fp8", "fp4", "nvfp4"])
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


# ------------------------------------------------------------------------------------------
# Clock samples inside the timed region; the peak a long timed region is compared with
# ------------------------------------------------------------------------------------------

def _line(sm, power, cap="Not Active", hw="Not Active"):
    return f"{sm}, 2070, {power}, 0x0, {hw}, Not Active, Not Active, {cap}"


def test_clock_summary_counts_only_samples_inside_the_timed_region():
    lines = [(0.0, _line(1980, 190)), (1.0, _line(1700, 1300, cap="Active")), (1.5, _line(1600, 1390, cap="Active")),
             (2.0, _line(1650, 1350)), (3.5, _line(1990, 200)), (3.6, "garbage")]
    c = bench.summarize_clocks(lines, (0.9, 2.1))
    assert c["samples"] == 5 and c["samples_under_load"] == 3
    assert c["sm_mhz"] == 1650 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    # no window: every sample counts, none is "under load"
    c = bench.summarize_clocks(lines, None)
    assert c["samples_under_load"] == 0 and c["sm_mhz"] == 1700


def test_clock_summary_reports_hardware_slowdown():
    c = bench.summarize_clocks([(1.0, _line(900, 700, hw="Active"))], (0.0, 2.0))
    assert c["reasons"] == ["hw_slowdown"]


def test_long_timed_regions_use_the_sustained_peak():
    peaks = {"bf16_tflops": 1933.3, "bf16_tflops_sustained": 1720.6, "hbm_gbs": 6775.3, "source": "measured"}
    w = W.NAMED["wide"]()
    short = bench.tensor_roofline(1600.0, w, peaks, 0.02)
    long = bench.tensor_roofline(1600.0, w, peaks, 2.1)
    assert short["peak"] == 1933.3 and "burst" in short["peak_source"]
    assert long["peak"] == 1720.6 and "sustained" in long["peak_source"]
    assert long["frac"] == pytest.approx(1600.0 / 1720.6)
    assert long["frac_vs_burst"] == pytest.approx(1600.0 / 1933.3)
    assert long["frac_vs_nominal"] == pytest.approx(1600.0 / 2250.0)
    f8 = bench.tensor_roofline(2400.0, W.NAMED["fp8"](), peaks, 2.1)
    assert f8["peak"] == pytest.approx(2 * 1720.6) and f8["frac_vs_nominal"] == pytest.approx(2400.0 / 4500.0)
    f4 = bench.tensor_roofline(4000.0, W.NAMED["fp4"](), peaks, 0.5)
    assert f4["peak"] == pytest.approx(6 * 1933.3)


def test_default_run_is_the_wide_hidden_workload_for_about_two_seconds():
    import argparse
    import inspect
    src = inspect.getsource(bench.main)
    assert 'default="wide"' in src and "default=2000" in src
    w = W.NAMED["wide"]()
    assert (w.num_experts, w.hidden, w.intermediate, w.accumulate, w.out_dtype) == (32, 7168, 2048, True, "bf16")
    # ~1.06 ms per call: 2000 steps keep the clock sampler (50 ms) busy for ~40 samples
    assert 2000 * 1.0e-3 >= 40 * bench.ClockSampler.INTERVAL_MS * 1e-3
    del argparse


def test_reference_steps_stay_bounded():
    class A:
        steps, warmup = 2000, 5
    assert bench.reference_budget(A) * (A.steps + A.warmup) <= 130
    A.steps, A.warmup = 2, 3
    assert bench.reference_budget(A) == 15.0


# ------------------------------------------------------------------------------------------
# Expert placement under torchrun (host side; the GPU path is per rank)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("world", [1, 2, 4, 8])
@pytest.mark.parametrize("name", ["wide", "skewed", "balanced"])
def test_rank_workloads_partition_every_layer_expert_once(name, world):
    w = W.NAMED[name]()
    parts = [bench.rank_workload(w, r, world) for r in range(world)]
    all_counts = np.concatenate([bench.layer_counts(w, l) for l in range(world)])
    assert sorted(np.concatenate([np.asarray(p.counts) for p in parts]).tolist()) == sorted(all_counts.tolist())
    sums = [p.tokens_sum for p in parts]
    assert sum(sums) == world * w.tokens_sum
    assert max(sums) - min(sums) <= int(np.max(all_counts))
    assert all(p.hidden == w.hidden and p.intermediate == w.intermediate and p.accumulate == w.accumulate
               and p.out_dtype == w.out_dtype and p.input_order == w.input_order for p in parts)
    if world == 1:
        assert parts[0] is w
    assert np.array_equal(bench.layer_counts(w, 0), np.asarray(w.counts))
