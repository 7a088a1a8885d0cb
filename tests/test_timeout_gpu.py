"""Failure detection without a GPU fault: a lost arrival ends the call with KGW_ERR_TIMEOUT.

The testing hook makes CTA 0's TMA producer skip one stage's arrival (and its copies), so the
MMA issuer's wait on that stage can never complete. Every wait in the kernel is bounded by a
wall-clock limit (set to 0.2 s here); the CTA that gives up drains its outstanding copies and
MMAs, frees its tensor memory and reports the timeout through status_dev. A normal call on the
same context afterwards must still be correct.
"""
import pytest
import torch

import workloads as W
from kgw_testlib import assert_close_to_oracle, ensure_built, oracle_full, run_gpu, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("hidden", [384, 512], ids=["single_cta_tiles", "cta_pair_tiles"])
def test_lost_arrival_times_out_and_context_stays_usable(hidden):
    kgw = ensure_built()
    # enough work items (16 experts x 24 or 16 tiles) that CTA 0 always claims some
    w = W.custom(16, hidden, 2048, [1024] * 16, seed=80)
    x = W.make_inputs(w, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    prev_t = kgw.kgw_debug_set(1, 200_000_000)
    prev_d = kgw.kgw_debug_set(2, 5)
    try:
        run_gpu(w, x, DEV, status=status)
        torch.cuda.synchronize()
    finally:
        kgw.kgw_debug_set(2, prev_d)
        kgw.kgw_debug_set(1, prev_t)
    assert int(status.item()) == kgw.KGW_ERR_TIMEOUT

    status.fill_(-1)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_OK
    ref, S = oracle_full(w, W.make_inputs(w, "cpu"))
    assert_close_to_oracle(w, to_f64(outs.stacked()), ref, S)
