"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The CUDA path computes every output; the oracle recomputes a sample of elements one by one
from the stored operands (row m of A_e, column n of B_e, in float64). The sample covers tile
corners of every non-empty expert plus uniformly drawn elements. Empty experts are checked
in full: zeros when overwriting, the pre-filled output bit for bit when accumulating.
"""
import numpy as np
import pytest
import torch

import oracle.kgw_oracle as O
import workloads as W
from kgw_testlib import bits8, bits16, ensure_built, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _samples(w, rng, n_uniform=300):
    counts = np.asarray(w.counts)
    nz = np.nonzero(counts)[0]
    out = []
    for e in nz[: min(len(nz), 24)]:
        for m in (0, 127, w.hidden - 1, w.hidden // 2 + 1):
            for n in (0, 255, w.intermediate - 1, w.intermediate // 2 + 3):
                out.append((int(e), m, n))
    for _ in range(n_uniform):
        out.append((int(rng.choice(nz)), int(rng.integers(w.hidden)), int(rng.integers(w.intermediate))))
    return out


def _check_full(w):
    kgw = ensure_built()
    x_cpu = W.make_inputs(w, "cpu")
    x = W.Inputs(*[None if t is None else t.to(DEV) for t in
                   (x_cpu.a, x_cpu.b, x_cpu.offsets, x_cpu.sfa, x_cpu.sfb, x_cpu.c)])
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact()
    bits = bits8 if (w.fp8 or w.fp4) else bits16
    a_bits, b_bits = bits(x_cpu.a), bits(x_cpu.b)
    offsets = x_cpu.offsets.numpy()
    sfa = None if x_cpu.sfa is None else x_cpu.sfa.numpy()
    sfb = None if x_cpu.sfb is None else x_cpu.sfb.numpy()
    rng = np.random.default_rng(1234)
    bad = []
    for (e, m, n) in _samples(w, rng):
        r, s = O.element_from_storage(a_bits, b_bits, offsets, w.hidden, w.intermediate, e, m, n,
                                      input_order=w.input_order, fp8=w.fp8, sfa=sfa, sfb=sfb,
                                      a_major=w.a_major, b_major=w.b_major, sf_format=w.sf_format, fp4=w.fp4)
        c = float(x_cpu.c[e, m, n].to(torch.float64)) if w.accumulate else 0.0
        ref = c + r
        got = float(outs.views[e][m, n].to(torch.float64).item())
        tol = float(O.tolerance(np.array(s), np.array(ref), w.out_dtype,
                                np.array(c) if (w.accumulate and w.out_dtype == "f32") else None))
        if not abs(got - ref) <= tol:
            bad.append((e, m, n, got, ref, tol))
    assert not bad, f"{len(bad)} sampled elements out of tolerance, first: {bad[:5]}"
    for e in np.nonzero(np.asarray(w.counts) == 0)[0]:
        if w.accumulate:
            assert torch.equal(outs.views[e], x.c[e]), f"empty expert {e} changed"
        else:
            assert not outs.views[e].any(), f"empty expert {e} not zero"


def test_full_balanced_bf16():
    _check_full(W.balanced())


def test_full_wide_accumulate_bf16():
    _check_full(W.wide())


def test_full_skewed_ragged_discrete():
    _check_full(W.skewed())


def test_full_fp8_blockscaled():
    kgw = ensure_built()
    if not kgw.lib():
        pytest.fail("library missing")
    _check_full(W.fp8())


def test_full_fp8_ue8m0_gran32():
    import dataclasses
    _check_full(dataclasses.replace(W.fp8(), sf_format="ue8m0_32"))


def test_full_balanced_token_major_a():
    """The balanced workload with A = dY^T read from dY stored token-major (M-major A)."""
    import dataclasses
    _check_full(dataclasses.replace(W.balanced(), a_major="mn"))


def test_full_fp4_blockscaled():
    """FP4 e2m1 operands with UE8M0 scales per 32 tokens, at the FP8 workload's shape."""
    _check_full(W.fp4())
