"""Benchmark of the K-grouped MoE weight-gradient GEMM on GB300.

One step = one call of the whole operation (plan kernel + persistent tcgen05 kernel) over one
batch of synthetic input: Wgrad[e] = A[:, begin_e:end_e] @ B[begin_e:end_e, :] for every
expert. Metric: TFLOP/s counting 2*hidden*intermediate*sum(n_e) FLOPs.

Default workload: BF16 wide-hidden, 32 experts, hidden 7168, intermediate 2048, per-expert tokens
round_to_256(2048*U(0.5,1.5)) with two experts set to 0 (seed 2), BF16 dense output pre-filled
N(0,1), accumulate: the largest of the configurations that fit one GPU. Its working set (A + B +
output, ~2.9 GB) is larger than L2, so no explicit flush is needed between steps. The default
2000 timed steps (~2 s) run long enough for the clock sampler (every 50 ms) to see the GPU under
sustained load; the roofline then uses the measured sustained bf16 peak.

Prints ONE JSON line (rank 0): the device-timed rate, the roofline of the main kernel (achieved
rate from CUDA events around each call, the measured peak, the DRAM bytes of one launch from the
committed ncu summary while the kernel source is unchanged), the end-to-end rate through the same
C entry point with pinned host inputs copied in and the result copied out every step (median of
five timed blocks), sampled clocks, and the float64 CPU oracle's rate on a bounded sample.
``--impl reference`` times the CPU oracle on the host cores instead (a bounded sample of the same
workload per step).

Other K-grouped workloads: ``--workload balanced|skewed|fp8|fp4|unaligned|fp8_unaligned|fp4_unaligned|tiny``. The M-grouped GEMM
(forward / dgrad of the same MoE layer, the masked decode layout, and their FP8 forms):
``--workload mg_forward|mg_dgrad|mg_masked|mg_fp8_forward|mg_fp8_masked|mg_tiny``, TFLOP/s
counting 2*N*K*(valid rows).

Multi-GPU (torchrun, N ranks): the job is the gradients of N MoE layers of the workload's shape
(layer 0 is the workload itself; layer l permutes its expert counts with seed + 1000*l), and the
N*E experts are placed on ranks by ``grouped_gemm_expert_gb300.partition.assign_experts``
(longest first, balanced token sums). Each rank computes its own experts from its own tokens with
no data-path exchange; timing is the max over ranks and the value counts all N layers: weak
scaling (the work per rank stays one layer's worth).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402
import workloads.mgrouped as MW  # noqa: E402

KERNEL_SOURCES = ["grouped_gemm_expert_gb300/csrc/kgw_kernels.cu", "grouped_gemm_expert_gb300/csrc/kgw_ptx.cuh",
                  "grouped_gemm_expert_gb300/csrc/kgw_internal.h"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background; each line is stamped with the host clock
    so that only the samples taken inside the timed region count as "under load"."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The host-clock window of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0,
                    "samples_under_load": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return summarize_clocks(self.lines, self.window)


def summarize_clocks(lines, window):
    """Median SM clock, maximum clock, active throttle reasons and sample counts.

    lines: [(host time, csv line)] in ClockSampler.FIELDS order. Samples stamped inside
    ``window`` (the timed region) are the ones under load; the median and the reasons come from
    them (from every sample when none falls inside).
    """
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    for t, ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm, smax, pw = float(parts[0]), float(parts[1]), float(parts[2])
        except ValueError:
            continue
        rows.append((t, sm, smax, pw, [nm for nm, v in zip(names, parts[4:8]) if v.lower() == "active"]))
    load = [r for r in rows if window and window[0] <= r[0] <= window[1]]
    use = load or rows
    reasons = sorted({nm for r in use for nm in r[4]})
    return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
            "sm_max_mhz": max(r[2] for r in rows) if rows else None,
            "power_w_median": statistics.median(r[3] for r in use) if use else None,
            "reasons": reasons, "samples": len(rows), "samples_under_load": len(load)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (a timing reduction, not part of the data path)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank processes its own batch (weak scaling), time is the max."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def traffic_record(workload: str):
    """DRAM bytes per launch of the main kernel from a committed ncu summary, if still current."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


def algorithmic_bytes(w) -> int:
    ts = w.tokens_sum
    counts = np.asarray(w.counts)
    blocks = int(np.sum(-(-counts // 128)))   # 128-token scale blocks of all experts (ts/128 when aligned)
    if w.fp4 and w.sf_format == "ue4m3_16":   # NVFP4: one UE4M3 byte per 16 tokens (a word per 64)
        b = (w.hidden + w.intermediate) * ts // 2 + (w.hidden + w.intermediate) * int(np.sum(-(-counts // 64))) * 4
    elif w.fp4:   # e2m1 two per byte, one UE8M0 byte per 32 tokens (a 4-byte word per 128-token block)
        b = (w.hidden + w.intermediate) * ts // 2 + (w.hidden + w.intermediate) * blocks * 4
    else:
        b = (w.hidden + w.intermediate) * ts * (1 if w.fp8 else 2)
    if w.fp8:
        b += (w.hidden + w.intermediate) * blocks * 4
    osz = 2 if w.out_dtype == "bf16" else 4
    nonempty = int((counts > 0).sum())
    if w.accumulate:
        b += 2 * nonempty * w.hidden * w.intermediate * osz
    else:
        b += w.num_experts * w.hidden * w.intermediate * osz
    return int(b)


NOMINAL_DENSE_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0, "fp4": 13500.0}
SUSTAINED_AFTER_S = 1.0   # a timed region at least this long is compared with the sustained peak


def tensor_roofline(achieved: float, w, peaks, timed_s: float) -> dict:
    """Roofline of a tensor-bound call: the measured bf16 peak (the sustained loop figure when the
    timed region lasts a second or more, else the burst), times the nominal dense ratio for FP8 (2)
    and FP4 (6); the fractions of the burst and of the nominal dense peak are reported beside it."""
    dt = "fp4" if getattr(w, "fp4", False) else ("fp8" if w.fp8 else "bf16")
    ratio = NOMINAL_DENSE_TFLOPS[dt] / NOMINAL_DENSE_TFLOPS["bf16"]
    sustained = timed_s >= SUSTAINED_AFTER_S and peaks.get("bf16_tflops_sustained")
    base = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak = base * ratio
    kind = "sustained" if sustained else "burst"
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": f"{peaks['source']} bf16 {kind}" + (f" x{ratio:g} (nominal dense ratio)" if ratio != 1 else "")
            + f", timed region {timed_s:.2f} s",
            "frac_vs_burst": achieved / (peaks["bf16_tflops"] * ratio),
            "frac_vs_nominal": achieved / NOMINAL_DENSE_TFLOPS[dt]}


def layer_counts(w, layer: int) -> np.ndarray:
    """Expert token counts of MoE layer ``layer`` of a multi-rank job: layer 0 is the workload's own
    counts, layer l a seeded permutation of them (the same count mix on other experts)."""
    counts = np.asarray(w.counts, dtype=np.int64)
    if layer == 0:
        return counts
    return counts[np.random.default_rng(w.seed + 1000 * layer).permutation(len(counts))]


def rank_workload(w, rank: int, world: int):
    """This rank's share of an N-layer job: the experts ``assign_experts`` places on it, as a local
    problem of the same shape and modes (its own tokens, drawn with a per-rank seed)."""
    import dataclasses

    from grouped_gemm_expert_gb300.partition import assign_experts

    if world == 1:
        return w
    all_counts = np.concatenate([layer_counts(w, l) for l in range(world)])
    mine = assign_experts(all_counts, world)[rank]
    if not mine:
        return None
    return dataclasses.replace(w, num_experts=len(mine), counts=all_counts[mine], seed=w.seed + 1000 * rank,
                               name=f"{w.name} [rank {rank} of {world}: {len(mine)} experts]")


def run_ours(args, w, rank, local, world):
    import grouped_gemm_expert_gb300 as kgw

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = W.make_inputs_device(w, dev)
    E, H, I = w.num_experts, w.hidden, w.intermediate
    odt = torch.bfloat16 if w.out_dtype == "bf16" else torch.float32
    if w.output_mode == "dense":
        out = torch.empty((E, H, I), dtype=odt, device=dev)
        outs_list = None
        ptrs = None
    else:
        outs_list = [torch.empty((H, I), dtype=odt, device=dev) for _ in range(E)]
        out = None
        ptrs = torch.tensor([t.data_ptr() for t in outs_list], dtype=torch.int64, device=dev)
    if w.accumulate:
        out.copy_(x.c)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kargs = kgw.make_args(E, H, I, w.tokens_sum, x.a, x.b, x.offsets, out=out, out_ptrs=ptrs,
                          out_dtype=kgw.KGW_OUT_BF16 if w.out_dtype == "bf16" else kgw.KGW_OUT_F32,
                          accumulate=w.accumulate,
                          input_order=kgw.KGW_RAGGED if w.input_order == "ragged" else kgw.KGW_TENSOR2D,
                          a_major=kgw.KGW_MN_MAJOR if w.a_major == "mn" else kgw.KGW_K_MAJOR,
                          b_major=kgw.KGW_K_MAJOR if w.b_major == "k" else kgw.KGW_MN_MAJOR,
                          status_dev=status)
    ws = kgw.workspace_for(kargs, w.fp8 or w.fp4, device=dev)
    stream = torch.cuda.current_stream()
    scaled = w.fp8 or w.fp4

    def call(args, sfa, sfb, s):
        if w.fp4 and w.unaligned:
            kgw.kgw_wgrad_fp4_unaligned(args, sfa, sfb, ws, stream=s)
        elif w.fp8 and w.unaligned:
            kgw.kgw_wgrad_fp8_unaligned(args, sfa, sfb, 1 if w.sf_format == "ue8m0_32" else 0, ws, stream=s)
        elif w.fp4 and w.sf_format == "ue4m3_16":
            kgw.kgw_wgrad_nvfp4(args, sfa, sfb, x.gsa, x.gsb, ws, stream=s)
        elif w.fp4:
            kgw.kgw_wgrad_fp4_ue8m0(args, sfa, sfb, ws, stream=s)
        elif w.fp8 and w.sf_format == "ue8m0_32":
            kgw.kgw_wgrad_fp8_ue8m0(args, sfa, sfb, ws, stream=s)
        elif w.fp8:
            kgw.kgw_wgrad_fp8_blockscaled(args, sfa, sfb, ws, stream=s)
        elif w.unaligned:
            kgw.kgw_wgrad_bf16_unaligned(args, ws, stream=s)
        else:
            kgw.kgw_wgrad_bf16(args, ws, stream=s)

    def step():
        call(kargs, x.sfa, x.sfb, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {kgw.kgw_status_string(int(status.item()))}")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.monotonic()
    t0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    if world > 1:
        torch.distributed.barrier()
    clocks.mark(h0, h1)
    clk = clocks.stop() if rank == 0 else None
    total_ms = t0.elapsed_time(t1)
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    timed_s = total_ms * 1e-3

    if args.no_e2e:
        return ms_per_step, per_launch_ms, None, 0, 0, clk, timed_s
    # ---- end to end through the public API, every step: the step's inputs are copied from
    # pinned host memory to the device, the call runs, and its result is copied back to pinned
    # host memory. Steps are pipelined over two buffer sets and three streams (copy-in, compute,
    # copy-out), so step i+1's upload and step i-1's download overlap step i's call.
    host_in = [t.cpu().pin_memory() for t in (x.a, x.b, x.offsets) + ((x.sfa, x.sfb) if scaled else ())]
    host_c = x.c.cpu().pin_memory() if w.accumulate else None
    h2d = sum(t.numel() * t.element_size() for t in host_in) + (
        host_c.numel() * host_c.element_size() if host_c is not None else 0)
    sets = []
    for _k in range(2):
        d_in = [torch.empty_like(t, device=dev) for t in host_in]
        if w.output_mode == "dense":
            d_out, d_list, d_ptrs = torch.empty((E, H, I), dtype=odt, device=dev), None, None
        else:
            d_list = [torch.empty((H, I), dtype=odt, device=dev) for _ in range(E)]
            d_out, d_ptrs = None, torch.tensor([t.data_ptr() for t in d_list], dtype=torch.int64, device=dev)
        ka = kgw.make_args(E, H, I, w.tokens_sum, d_in[0], d_in[1], d_in[2], out=d_out, out_ptrs=d_ptrs,
                           out_dtype=kargs.out_dtype, accumulate=w.accumulate, input_order=kargs.input_order,
                           a_major=kargs.a_major, b_major=kargs.b_major, status_dev=status)
        h_out = torch.empty((E, H, I), dtype=odt).pin_memory()
        sets.append(dict(d_in=d_in, d_out=d_out, d_list=d_list, args=ka, h_out=h_out,
                         ev_in=torch.cuda.Event(), ev_comp=torch.cuda.Event(), ev_out=torch.cuda.Event()))
    d2h = sets[0]["h_out"].numel() * sets[0]["h_out"].element_size()
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    started = [False, False]

    def e2e_step(i):
        k = i % 2
        S = sets[k]
        with torch.cuda.stream(s_in):
            if started[k]:
                s_in.wait_event(S["ev_comp"])   # the call that read this set's inputs is done
                s_in.wait_event(S["ev_out"])    # and its result has been copied out
            for d, h in zip(S["d_in"], host_in):
                d.copy_(h, non_blocking=True)
            if host_c is not None:
                S["d_out"].copy_(host_c, non_blocking=True)
            S["ev_in"].record(s_in)
        s_comp.wait_event(S["ev_in"])
        call(S["args"], S["d_in"][3] if scaled else None, S["d_in"][4] if scaled else None, s_comp)
        S["ev_comp"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(S["ev_comp"])
            if S["d_out"] is not None:
                S["h_out"].copy_(S["d_out"], non_blocking=True)
            else:
                for e in range(E):
                    S["h_out"][e].copy_(S["d_list"][e], non_blocking=True)
            S["ev_out"].record(s_out)
        started[k] = True

    # the host link is shared with whatever else the machine runs: time five blocks of steps and
    # report the median block
    e2e_steps = max(4, min(args.steps, 10))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    blocks = []
    for _rep in range(5):
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        blocks.append(e0.elapsed_time(e1) / e2e_steps)
    e2e_ms = max_over_ranks(statistics.median(blocks), world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {kgw.kgw_status_string(int(status.item()))}")
    return ms_per_step, per_launch_ms, e2e_ms, h2d, d2h, clk, timed_s


def mg_algorithmic_bytes(w) -> int:
    """A's valid rows, every non-empty group's weight, and D's valid rows (read too if accumulating);
    FP8 adds the scales of those rows and columns (one word per 128 K)."""
    counts = np.asarray(w.counts)
    osz = {"f32": 4, "bf16": 2, "f16": 2}[w.out_dtype]
    esz = 1 if w.fp8 else 2
    rows = int(counts.sum())
    groups = int((counts > 0).sum())
    b = rows * w.k * esz + groups * w.n * w.k * esz + rows * w.n * osz * (2 if w.accumulate else 1)
    if w.fp8:
        b += (rows + groups * w.n) * (w.k // 128) * 4
    return int(b)


def run_ours_mg(args, w, rank, local, world):
    """Device-timed steps and the end-to-end leg for an M-grouped workload."""
    import dataclasses

    import grouped_gemm_expert_gb300 as kgw

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = MW.make_mg_inputs(dataclasses.replace(w, seed=w.seed + 1000 * rank), dev, on_device_rng=True)
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.out_dtype]
    d_shape = (w.num_groups, w.max_m, w.n) if w.layout == "masked" else (w.rows, w.n)
    d = torch.zeros(d_shape, dtype=odt, device=dev) if x.d0 is None else x.d0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lay = {"offsets": kgw.KGW_MG_OFFSETS, "indices": kgw.KGW_MG_INDICES, "masked": kgw.KGW_MG_MASKED}[w.layout]
    fmt = 1 if w.sf_format == "ue8m0_32" else 0
    mk = lambda a, b, g, dd: kgw.make_mgrouped_args(
        w.num_groups, w.m, w.n, w.k, a, b, g, dd, layout=lay,
        b_major=kgw.KGW_K_MAJOR if w.b_major == "k" else kgw.KGW_MN_MAJOR,
        out_dtype={"f32": kgw.KGW_OUT_F32, "bf16": kgw.KGW_OUT_BF16, "f16": kgw.KGW_OUT_F16}[w.out_dtype],
        accumulate=w.accumulate, status_dev=status)
    kargs = mk(x.a, x.b, x.groups, d)
    ws = torch.empty(kgw.kgw_mgrouped_workspace_size(kargs), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # the masked decode workload (~0.3 GB) fits in L2: flush it between steps with a 256 MB write
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if w.layout == "masked" else None

    def call(args, sfa, sfb):
        if w.fp8:
            kgw.kgw_mgrouped_fp8(args, sfa, sfb, fmt, ws, stream=stream)
        else:
            kgw.kgw_mgrouped_bf16(args, ws, stream=stream)

    def step():
        if flush is not None:
            flush.fill_(1)
        call(kargs, x.sfa, x.sfb)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {kgw.kgw_status_string(int(status.item()))}")
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    h0 = time.monotonic()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(1)
        starts[i].record(stream)
        call(kargs, x.sfa, x.sfb)
        ends[i].record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    if world > 1:
        torch.distributed.barrier()
    clocks.mark(h0, h1)
    clk = clocks.stop() if rank == 0 else None
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # a step is the call; the L2 flush between calls is not part of it
    ms_per_step = max_over_ranks(statistics.mean(per_launch_ms), world, dev)
    timed_s = h1 - h0
    if args.no_e2e:
        return ms_per_step, per_launch_ms, None, 0, 0, clk, timed_s
    # end to end: inputs from pinned host memory, the call, D back to pinned host memory (serial)
    host_in = [t.cpu().pin_memory() for t in (x.a, x.b, x.groups) + ((x.sfa, x.sfb) if w.fp8 else ())]
    host_d0 = None if x.d0 is None else x.d0.cpu().pin_memory()
    d_in = [torch.empty_like(t, device=dev) for t in host_in]
    d_out = torch.empty_like(d)
    h_out = torch.empty(d.shape, dtype=odt).pin_memory()
    ea = mk(d_in[0], d_in[1], d_in[2], d_out)
    h2d = sum(t.numel() * t.element_size() for t in host_in) + (0 if host_d0 is None else host_d0.numel() * host_d0.element_size())
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        for dd, h in zip(d_in, host_in):
            dd.copy_(h, non_blocking=True)
        if host_d0 is not None:
            d_out.copy_(host_d0, non_blocking=True)
        call(ea, d_in[3] if w.fp8 else None, d_in[4] if w.fp8 else None)
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 8))
    blocks = []
    for _rep in range(5):  # median of five blocks, as for the K-grouped leg
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        blocks.append(e0.elapsed_time(e1) / n)
    e2e_ms = max_over_ranks(statistics.median(blocks), world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {kgw.kgw_status_string(int(status.item()))}")
    return ms_per_step, per_launch_ms, e2e_ms, h2d, d2h, clk, timed_s


class MgOracleSampler:
    """The float64 M-grouped oracle, as it stands, on the host cores: the operands are decoded once,
    then ``run`` evaluates the oracle on blocks of up to 512 rows of one group at a time (each a
    single-group problem through the oracle's own entry point) until a time budget is spent."""
    ROWS = 512

    def __init__(self, w):
        import oracle.kgw_oracle as O
        import oracle.mgrouped_oracle as MO

        self.w, self.MO = w, MO
        x = MW.make_mg_inputs(w, "cpu")
        if w.fp8:
            u8 = lambda t: t.contiguous().view(torch.uint8).numpy()
            self.A, self.B = MO.dequantize_fp8(u8(x.a), u8(x.b), x.sfa.numpy(), x.sfb.numpy(), w.b_major, w.sf_format)
        else:
            self.A = O.bf16_to_f64(x.a.contiguous().view(torch.int16).numpy().view(np.uint16)).reshape(-1, w.k)
            self.B = O.bf16_to_f64(x.b.contiguous().view(torch.int16).numpy().view(np.uint16))
        groups = x.groups.numpy()
        self.units = [(g, r[i:i + self.ROWS]) for g, r in enumerate(MO.group_rows(w.layout, groups, w.m, w.num_groups))
                      for i in range(0, len(r), self.ROWS)]
        self.next = 0

    def run(self, budget_s: float):
        """(TFLOP/s, seconds, units done): at least one unit, then more until ``budget_s``."""
        w = self.w
        flops, done = 0.0, 0
        t0 = time.perf_counter()
        while done == 0 or time.perf_counter() - t0 < budget_s:
            g, r = self.units[self.next % len(self.units)]
            self.next += 1
            self.MO.mgrouped(self.A[r], self.B[g:g + 1], "offsets", [len(r)], len(r), b_major=w.b_major,
                             with_bound=False)
            flops += 2.0 * len(r) * w.n * w.k
            done += 1
        dt = time.perf_counter() - t0
        return flops / dt / 1e12, dt, done


def reference_budget(args) -> float:
    """Seconds of oracle work per reference step, so that warm-up plus timed steps take ~2 minutes."""
    return max(0.05, min(15.0, 120.0 / max(1, args.steps + args.warmup)))


def main_mg(args, world, rank, local):
    w = MW.MG_NAMED[args.workload]()
    flops = w.flops
    metric = "M-grouped GEMM TFLOP/s (2*N*K*valid rows)"
    config = {"workload": w.name, "groups": w.num_groups, "layout": w.layout, "m": w.m, "n": w.n, "k": w.k,
              "valid_rows": w.valid_rows, "b_major": w.b_major, "output": w.out_dtype, "accumulate": w.accumulate,
              "l2": "L2 flushed (256 MB write) between steps" if w.layout == "masked"
              else "inputs larger than L2 (no flush needed)",
              "parallelism": "single GPU" if world == 1 else f"replica x{world} (one batch per rank)"}
    if args.impl == "reference":
        if rank != 0:
            return
        sampler = MgOracleSampler(w)
        budget = reference_budget(args)
        rates = []
        for i in range(args.warmup + args.steps):
            r, dt, done = sampler.run(budget)
            if i >= args.warmup:
                rates.append((r, dt, done))
        val = statistics.median(r for r, _, _ in rates)
        ms = statistics.median(dt for _, dt, _ in rates) * 1e3
        print(json.dumps({"impl": "reference", "metric": metric, "value": val, "unit": "TFLOP/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                           "sample": f"float64 oracle over blocks of up to {MgOracleSampler.ROWS} rows of one group, "
                                                     f"{ms / 1e3:.2f} s per step"},
                          "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    ms_per_step, per_launch, e2e_ms, h2d, d2h, clk, timed_s = run_ours_mg(args, w, rank, local, world)
    value = job_throughput(flops, ms_per_step, world)
    peaks = measured_peaks()
    launch_ms = statistics.mean(per_launch)
    achieved = flops / (launch_ms * 1e-3) / 1e12
    abytes = mg_algorithmic_bytes(w)
    # below the ridge point (few rows per group: the decode case) the weights' HBM reads bound it
    troof = tensor_roofline(achieved, w, peaks, timed_s)
    hbm_bound = flops / abytes < troof["peak"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": abytes / (launch_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"{peaks['source']} HBM copy"}
    else:
        roof = troof
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": traffic_record(args.workload),
                 "algorithmic_bytes": abytes, "flops": flops,
                 "kernel": "wgrad_kernel M-grouped instantiation (+ plan_mgrouped_kernel)"})
    line = {"metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8" if w.fp8 else "bf16", "data": "synthetic", "config": config,
            "roofline": roof,
            "e2e": None if e2e_ms is None else {"value": job_throughput(flops, e2e_ms, world), "unit": "TFLOP/s",
                                                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * args.steps, "clocks": clk}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, dt, done = MgOracleSampler(w).run(args.cpu_budget)
        line["cpu_baseline"] = {"value": r, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"float64 oracle, {done} blocks of up to {MgOracleSampler.ROWS} rows of one "
                                          f"group of the same workload, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


class OracleSampler:
    """The float64 oracle, as it stands, on the host cores: the operands are decoded (and scaled)
    once, then ``run`` evaluates the oracle's ``wgrad`` on blocks of up to 512 rows of A_e for one
    expert at a time (the same definition on a row block) until a time budget is spent."""
    ROWS = 512

    def __init__(self, w):
        import oracle.kgw_oracle as O

        self.w, self.O = w, O
        x = W.make_inputs(w, "cpu")
        bits = (lambda t: t.contiguous().view(torch.uint8).numpy()) if (w.fp8 or w.fp4) else \
            (lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16))
        a_bits, b_bits = bits(x.a), bits(x.b)
        del x.a, x.b
        dec = O.e2m1_to_f64 if w.fp4 else (O.e4m3_to_f64 if w.fp8 else O.bf16_to_f64)
        A = O.logical_a(dec(a_bits), w.hidden, w.offsets, w.input_order, w.a_major)
        B = O.logical_b(dec(b_bits), w.intermediate, w.offsets, w.input_order, w.b_major)
        if w.fp8 or w.fp4:
            sa, blk = O.decode_scales(x.sfa.numpy(), w.sf_format)
            sb, _ = O.decode_scales(x.sfb.numpy(), w.sf_format)
            rows = O.token_scale_rows(w.offsets, blk)
            A = O.apply_scales_rows(A, sa, blk, rows)
            B = O.apply_scales_cols(B, sb, blk, rows)
        self.A, self.B = A, B
        self.units = [(b, end, r0) for (b, end) in O.expert_ranges(w.offsets) if end > b
                      for r0 in range(0, w.hidden, self.ROWS)]
        self.next = 0

    def run(self, budget_s: float):
        """(TFLOP/s, seconds, units done): at least one unit, then more until ``budget_s``."""
        w, O = self.w, self.O
        flops, done = 0.0, 0
        t0 = time.perf_counter()
        while done == 0 or time.perf_counter() - t0 < budget_s:
            b, end, r0 = self.units[self.next % len(self.units)]
            self.next += 1
            r1 = min(w.hidden, r0 + self.ROWS)
            O.wgrad(self.A[r0:r1, b:end], self.B[b:end, :], np.array([end - b], dtype=np.int64), with_bound=False)
            flops += 2.0 * (r1 - r0) * w.intermediate * (end - b)
            done += 1
        dt = time.perf_counter() - t0
        return flops / dt / 1e12, dt, done


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max((i.get("num_threads", 0) for i in info), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wide", choices=sorted(W.NAMED) + sorted(MW.MG_NAMED))
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    if args.workload in MW.MG_NAMED:
        main_mg(args, world, rank, local)
        return
    w = W.NAMED[args.workload]()
    flops = w.flops
    config = {"workload": w.name, "experts": w.num_experts, "hidden": w.hidden, "intermediate": w.intermediate,
              "tokens_sum": w.tokens_sum, "input_order": w.input_order, "output": f"{w.output_mode} {w.out_dtype}",
              "accumulate": w.accumulate, "l2": "inputs larger than L2 (no flush needed)",
              "parallelism": "single GPU" if world == 1 else
              f"expert-parallel x{world}: {world} layers' experts placed longest-first on {world} ranks"}
    if w.tokens_sum * (w.hidden + w.intermediate) * 2 < 129e6:
        config["l2"] = "working set fits L2 (warm)"

    if args.impl == "reference":
        if rank != 0:
            return
        sampler = OracleSampler(w)
        budget = reference_budget(args)
        rates = []
        for i in range(args.warmup + args.steps):
            r, dt, done = sampler.run(budget)
            if i >= args.warmup:
                rates.append((r, dt, done))
        val = statistics.median(r for r, _, _ in rates)
        ms = statistics.median(dt for _, dt, _ in rates) * 1e3
        line = {"impl": "reference", "metric": "K-grouped wgrad TFLOP/s (2*H*I*sum n_e)", "value": val,
                "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                 "sample": f"float64 oracle over blocks of up to {OracleSampler.ROWS} rows of one "
                                           f"expert's product (cycling through the workload), {ms / 1e3:.2f} s per step"},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    wl = rank_workload(w, rank, world)
    if wl is None:
        raise RuntimeError(f"rank {rank} was assigned no experts")
    ms_per_step, per_launch, e2e_ms, h2d, d2h, clk, timed_s = run_ours(args, wl, rank, local, world)
    # every layer has the workload's token sum: the job's FLOPs are world x the workload's
    value = job_throughput(flops, ms_per_step, world)
    peaks = measured_peaks()
    launch_ms = statistics.mean(per_launch)
    achieved = wl.flops / (launch_ms * 1e-3) / 1e12
    roof = tensor_roofline(achieved, w, peaks, timed_s)
    traffic = traffic_record(args.workload) if world == 1 else None
    line = {"metric": "K-grouped wgrad TFLOP/s (2*H*I*sum n_e)", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp4" if w.fp4 else ("fp8" if w.fp8 else "bf16"), "data": "synthetic", "config": config,
            "roofline": dict(roof, traffic=traffic, algorithmic_bytes=algorithmic_bytes(wl),
                             kernel="wgrad_kernel (+ plan_kernel, a few us, inside the same events)"),
            "e2e": None if e2e_ms is None else {"value": job_throughput(flops, e2e_ms, world), "unit": "TFLOP/s",
                                                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * args.steps,
            "clocks": clk}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, dt, done = OracleSampler(w).run(args.cpu_budget)
        line["cpu_baseline"] = {"value": r, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"float64 oracle, {done} blocks of up to {OracleSampler.ROWS} rows of one "
                                          f"expert's product of the same workload, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
