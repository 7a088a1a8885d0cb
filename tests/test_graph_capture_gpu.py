"""The K-grouped calls read the offsets on the device and never synchronise with the host, so a
call can be captured in a CUDA graph once and replayed with new per-expert counts (same
tokens_sum) and new operand values written into the same buffers. Every replay is compared with
the float64 oracle for the counts and values it saw."""
import numpy as np
import pytest
import torch

import workloads as W
from kgw_testlib import Outputs, assert_close_to_oracle, ensure_built, oracle_full, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("kind", ["bf16", "bf16_pair_split", "fp8", "unaligned"])
def test_captured_call_replays_with_new_counts(kind):
    kgw = ensure_built()
    if kind == "bf16":
        counts_seq = [[512, 256, 0, 768], [256, 1024, 256, 0], [0, 0, 1536, 0]]
        mk = lambda c, seed: W.custom(4, 256, 512, c, seed=seed, out_dtype="bf16")
    elif kind == "bf16_pair_split":
        counts_seq = [[8192, 256, 0, 512], [256, 512, 8192, 0]]
        mk = lambda c, seed: W.custom(4, 512, 256, c, seed=seed)
    elif kind == "fp8":
        counts_seq = [[512, 256, 0, 768], [768, 0, 512, 256]]
        mk = lambda c, seed: W.custom(4, 256, 512, c, seed=seed, fp8=True, out_dtype="bf16")
    else:
        counts_seq = [[8, 600, 0, 928], [1000, 24, 512, 0]]
        mk = lambda c, seed: W.custom(4, 256, 512, c, seed=seed, unaligned=True)
    w0 = mk(counts_seq[0], 150)
    x = W.make_inputs(w0, DEV)
    outs = Outputs(w0, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(w0.num_experts, w0.hidden, w0.intermediate, w0.tokens_sum, x.a, x.b, x.offsets,
                         out=outs.dense, out_dtype=kgw.KGW_OUT_BF16 if w0.out_dtype == "bf16" else kgw.KGW_OUT_F32,
                         status_dev=status)
    ws = kgw.workspace_for(args, w0.fp8, device=DEV)
    s = torch.cuda.Stream()

    def call(stream):
        if w0.fp8:
            kgw.kgw_wgrad_fp8_blockscaled(args, x.sfa, x.sfb, ws, stream=stream)
        elif w0.unaligned:
            kgw.kgw_wgrad_bf16_unaligned(args, ws, stream=stream)
        else:
            kgw.kgw_wgrad_bf16(args, ws, stream=stream)

    with torch.cuda.stream(s):
        call(s)                      # first call outside the capture (one-time host set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    for i, counts in enumerate(counts_seq):
        w = mk(counts, 151 + i)
        xi = W.make_inputs(w, "cpu")
        x.a.copy_(xi.a)
        x.b.copy_(xi.b)
        x.offsets.copy_(xi.offsets)
        if w.fp8:
            x.sfa.copy_(xi.sfa)
            x.sfb.copy_(xi.sfb)
        outs.dense.fill_(7.25)
        status.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
        assert outs.guards_intact()
        ref, S = oracle_full(w, xi)
        assert_close_to_oracle(w, to_f64(outs.stacked()), ref, S)
        for e in np.nonzero(np.asarray(counts) == 0)[0]:
            assert not outs.views[e].any(), f"replay {i}: empty expert {e} not zero"
