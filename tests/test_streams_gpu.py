"""Calls on different streams, each with its own workspace, may run at the same time: the library
keeps no per-call state outside the caller's workspace (the scheduler's item counter, the plan, the
per-expert descriptors and the split-K partials all live there). Three different calls are queued
on three streams several times over, so that their kernels overlap on the GPU; every result must be
bitwise identical to the same call run alone (the kernels are deterministic, and each call
overwrites its whole output)."""
import pytest
import torch

import workloads as W
import workloads.mgrouped as MW
from kgw_testlib import Outputs, ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _k_grouped(kgw, w):
    x = W.make_inputs(w, DEV)
    outs = Outputs(w, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(w.num_experts, w.hidden, w.intermediate, w.tokens_sum, x.a, x.b, x.offsets,
                         out=outs.dense, out_dtype=kgw.KGW_OUT_BF16 if w.out_dtype == "bf16" else kgw.KGW_OUT_F32,
                         status_dev=status)
    ws = kgw.workspace_for(args, w.fp8, device=DEV)

    def call(stream):
        if w.fp8:
            kgw.kgw_wgrad_fp8_blockscaled(args, x.sfa, x.sfb, ws, stream=stream)
        else:
            kgw.kgw_wgrad_bf16(args, ws, stream=stream)

    return call, outs.dense, status, (x, outs, args, ws)


def _m_grouped(kgw, w):
    x = MW.make_mg_inputs(w, DEV)
    d = torch.full((w.rows, w.n), 7.25, dtype=torch.bfloat16, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_mgrouped_args(w.num_groups, w.m, w.n, w.k, x.a, x.b, x.groups, d, status_dev=status)
    ws = torch.empty(kgw.kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=DEV)

    def call(stream):
        kgw.kgw_mgrouped_bf16(args, ws, stream=stream)

    return call, d, status, (x, args, ws)


def test_concurrent_streams_match_serial():
    kgw = ensure_built()
    calls = [
        # K-grouped BF16 on CTA pairs with one long expert (split along K), FP32 out
        _k_grouped(kgw, W.custom(4, 512, 512, [8192, 256, 0, 1024], seed=170)),
        # K-grouped FP8, BF16 out
        _k_grouped(kgw, W.custom(4, 256, 512, [512, 768, 256, 0], seed=171, fp8=True, out_dtype="bf16")),
        # M-grouped BF16 forward
        _m_grouped(kgw, MW.mg_custom(4, 512, 256, "offsets", [256, 512, 0, 384], seed=172)),
    ]
    torch.cuda.synchronize()
    alone = []
    for call, out, status, _ in calls:
        call(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
        alone.append(out.clone())
    for _, out, status, _ in calls:
        out.fill_(7.25)
        status.fill_(-1)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in calls]
    for _ in range(4):
        for (call, _, _, _), s in zip(calls, streams):
            call(s)
    torch.cuda.synchronize()
    for i, ((_, out, status, _), ref) in enumerate(zip(calls, alone)):
        assert int(status.item()) == 0, (i, kgw.kgw_status_string(int(status.item())))
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8)), f"call {i} differs when run concurrently"
