"""The largest supported expert / group counts (4096) on the GPU.

K-grouped: 4096 experts, one in sixteen with 256 tokens; every empty expert's output must be zero
(checked in full on the device), every element of the others against the oracle computed one
expert at a time. M-grouped: 4096 groups, one in thirty-two with 128 rows, against the full
oracle. Tolerance as in the other parity tests.
"""
import numpy as np
import pytest
import torch

import oracle.kgw_oracle as O
import oracle.mgrouped_oracle as MO
import workloads as W
import workloads.mgrouped as MW
from kgw_testlib import bits16, ensure_built, run_gpu, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_max_experts_k_grouped():
    kgw = ensure_built()
    E = 4096
    counts = np.where(np.arange(E) % 16 == 5, 256, 0)
    w = W.custom(E, 128, 256, counts, seed=160, out_dtype="bf16")
    x_cpu = W.make_inputs(w, "cpu")
    x = W.Inputs(x_cpu.a.to(DEV), x_cpu.b.to(DEV), x_cpu.offsets.to(DEV))
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact()
    empty = torch.from_numpy(counts == 0).to(DEV)
    assert not outs.dense[empty].any(), "an empty expert's output is not zero"
    a_bits, b_bits = bits16(x_cpu.a), bits16(x_cpu.b)
    bad = []
    for e in np.nonzero(counts)[0]:
        r, s = O.expert_from_storage(a_bits, b_bits, w.offsets, 128, 256, int(e))
        got = to_f64(outs.dense[e])
        tol = O.tolerance(s, r, "bf16")
        if not np.all(np.abs(got - r) <= tol):
            bad.append(int(e))
    assert not bad, f"experts out of tolerance: {bad[:8]}"


def test_max_experts_k_grouped_accumulate():
    """4096 experts accumulating into BF16, one in sixteen with 256 tokens: the empty experts have
    no work items (their prefix sums repeat, so the scheduler's expert search crosses runs of
    fifteen equal entries), their outputs must stay bit-identical, and every element of the
    others must match C + the oracle's product."""
    kgw = ensure_built()
    E = 4096
    counts = np.where(np.arange(E) % 16 == 5, 256, 0)
    w = W.custom(E, 128, 256, counts, seed=161, out_dtype="bf16", accumulate=True)
    x_cpu = W.make_inputs(w, "cpu")
    x = W.Inputs(x_cpu.a.to(DEV), x_cpu.b.to(DEV), x_cpu.offsets.to(DEV), c=x_cpu.c.to(DEV))
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact()
    empty = torch.from_numpy(counts == 0).to(DEV)
    assert torch.equal(outs.dense[empty].view(torch.int16), x.c[empty].view(torch.int16)), \
        "an empty expert's accumulated output changed"
    a_bits, b_bits = bits16(x_cpu.a), bits16(x_cpu.b)
    c64 = x_cpu.c.to(torch.float64).numpy()
    bad = []
    for e in np.nonzero(counts)[0]:
        r, s = O.expert_from_storage(a_bits, b_bits, w.offsets, 128, 256, int(e))
        ref = c64[e] + r
        got = to_f64(outs.dense[e])
        tol = O.tolerance(s, ref, "bf16")
        if not np.all(np.abs(got - ref) <= tol):
            bad.append(int(e))
    assert not bad, f"experts out of tolerance: {bad[:8]}"


def test_max_groups_m_grouped():
    kgw = ensure_built()
    G = 4096
    counts = np.where(np.arange(G) % 32 == 7, 128, 0)
    w = MW.mg_custom(G, 256, 64, "offsets", counts, seed=162, out_dtype="f32")
    x_cpu = MW.make_mg_inputs(w, "cpu")
    x = MW.make_mg_inputs(w, DEV)
    d = torch.full((w.rows, w.n), 7.25, dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    kgw.mgrouped(x.a, x.b, x.groups, d=d, out_dtype="f32", status_dev=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    ref, S = MO.mgrouped_from_storage(bits16(x_cpu.a), bits16(x_cpu.b), "offsets", x_cpu.groups.numpy(), w.m,
                                      d_init=np.zeros((w.rows, w.n)))
    tol = O.tolerance(S, ref, "f32")
    assert np.all(np.abs(to_f64(d) - ref) <= tol)
