"""The entry point that allocates nothing (kgw_wgrad_bf16_noalloc), checked through the C ABI.

Some callers cannot allocate device memory when they call: a framework whose caching
allocator owns the device memory, a runtime that forbids allocation after start-up, or a
plug-in that only receives tensors and a stream. For them the library keeps its scratch in a
static device array. This test compares that entry point with kgw_wgrad_bf16 (workspace
entry point) on two calls in a row, within the same per-element tolerance as the parity tests.
It lives in its own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from kgw_testlib import Outputs, ensure_built, oracle_full, run_gpu, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(kgw, w, x, status):
    outs = Outputs(w, DEV, x.c)
    args = kgw.make_args(w.num_experts, w.hidden, w.intermediate, w.tokens_sum, x.a, x.b, x.offsets,
                         out=outs.dense, out_ptrs=outs.ptrs,
                         out_dtype=kgw.KGW_OUT_BF16 if w.out_dtype == "bf16" else kgw.KGW_OUT_F32,
                         accumulate=w.accumulate,
                         input_order=kgw.KGW_RAGGED if w.input_order == "ragged" else kgw.KGW_TENSOR2D,
                         status_dev=status)
    stream = torch.cuda.current_stream().cuda_stream
    rc = kgw.lib().kgw_wgrad_bf16_noalloc(ctypes.byref(args), ctypes.c_void_p(stream))
    assert rc == kgw.KGW_OK, kgw.kgw_status_string(rc)
    return outs


def _compare(w, got, want, x_cpu):
    """Both entry points within the parity tolerance of the oracle, and of each other.

    The static scratch holds fewer split-K partial tiles than a full workspace, so a long expert
    may be summed in a different order; each result then carries its own final rounding (one
    BF16 ulp can separate them), so two results that each meet the bound differ by at most twice it.
    """
    import oracle.kgw_oracle as O
    ref, S = oracle_full(w, x_cpu)
    c = to_f64(x_cpu.c) if (w.accumulate and w.out_dtype == "f32") else None
    tol = O.tolerance(S, ref, w.out_dtype, c)
    g, wnt = to_f64(got), to_f64(want)
    assert np.all(np.abs(g - ref) <= tol), "no-alloc entry point out of tolerance"
    assert np.all(np.abs(wnt - ref) <= tol), "workspace entry point out of tolerance"
    diff = np.abs(g - wnt)
    assert np.all(diff <= 2 * tol), f"max diff {diff.max():.3g}, worst diff/tol {(diff / tol).max():.3g}"


CASES = [
    # split-K on the long expert, so the static scratch's partial tiles and counters are used
    W.custom(3, 256, 512, [8192, 0, 768], seed=71),
    # a different shape, ragged input, accumulate into BF16: must not see the previous call's state
    W.custom(5, 384, 768, [512, 256, 0, 2304, 4096], seed=72, input_order="ragged", accumulate=True,
             out_dtype="bf16"),
]


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    kgw = ensure_built()
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for w in CASES:
        x_cpu = W.make_inputs(w, "cpu")
        x = W.make_inputs(w, DEV)
        want = run_gpu(w, x, DEV).stacked().clone()
        got_outs = _noalloc(kgw, w, x, status)
        torch.cuda.synchronize()
        assert int(status.item()) == kgw.KGW_OK
        assert got_outs.guards_intact()
        _compare(w, got_outs.stacked(), want, x_cpu)

