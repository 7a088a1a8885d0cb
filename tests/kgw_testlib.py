"""Shared helpers for the tests: build/load the library, run the CUDA path, compare with the oracle."""
import os
import re
import subprocess
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kgw.h")


def ensure_built():
    import grouped_gemm_expert_gb300 as kgw
    if not os.path.exists(kgw.LIB_PATH):
        from grouped_gemm_expert_gb300 import build
        build.build()
    return kgw


def header_functions():
    """Names of the functions include/kgw.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(kgw_\w+)\s*\(", src, flags=re.M)))


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


class Outputs:
    """Output buffers with guard bands (canaries) around them to catch out-of-bounds writes."""
    GUARD = 4096  # elements

    def __init__(self, w, device, c_init=None):
        self.w = w
        dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.out_dtype]
        E, H, I = w.num_experts, w.hidden, w.intermediate
        self.dtype = dt
        g = self.GUARD
        if w.output_mode == "dense":
            self.buf = torch.full((E * H * I + 2 * g,), 7.25, dtype=dt, device=device)
            self.views = [self.buf[g + e * H * I: g + (e + 1) * H * I].view(H, I) for e in range(E)]
            self.dense = self.buf[g:g + E * H * I].view(E, H, I)
            self.ptrs = None
        else:
            self.bufs = [torch.full((H * I + 2 * g,), 7.25, dtype=dt, device=device) for _ in range(E)]
            self.views = [b[g:g + H * I].view(H, I) for b in self.bufs]
            self.dense = None
            self.ptrs = torch.tensor([v.data_ptr() for v in self.views], dtype=torch.int64, device=device)
        if c_init is not None:
            for e in range(E):
                self.views[e].copy_(c_init[e])

    def guards_intact(self) -> bool:
        g = self.GUARD
        bufs = [self.buf] if self.w.output_mode == "dense" else self.bufs
        for b in bufs:
            if not (torch.all(b[:g] == 7.25) and torch.all(b[-g:] == 7.25)):
                return False
        return True

    def stacked(self) -> torch.Tensor:
        return torch.stack([v for v in self.views])


def run_gpu(w, x, device="cuda", status=None, workspace=None, outputs=None):
    """Run the CUDA path for workload ``w`` on inputs ``x`` (already on ``device``)."""
    kgw = ensure_built()
    outs = outputs or Outputs(w, device, x.c)
    args = kgw.make_args(w.num_experts, w.hidden, w.intermediate, w.tokens_sum, x.a, x.b, x.offsets,
                         out=outs.dense, out_ptrs=outs.ptrs,
                         out_dtype={"bf16": kgw.KGW_OUT_BF16, "f16": kgw.KGW_OUT_F16}.get(w.out_dtype, kgw.KGW_OUT_F32),
                         accumulate=w.accumulate,
                         input_order=kgw.KGW_RAGGED if w.input_order == "ragged" else kgw.KGW_TENSOR2D,
                         a_major=kgw.KGW_MN_MAJOR if w.a_major == "mn" else kgw.KGW_K_MAJOR,
                         b_major=kgw.KGW_K_MAJOR if w.b_major == "k" else kgw.KGW_MN_MAJOR,
                         status_dev=status)
    if workspace is None:
        workspace = kgw.workspace_for(args, w.fp8 or w.fp4, device=device)
    if w.fp4 and w.sf_format == "ue4m3_16":
        kgw.kgw_wgrad_nvfp4(args, x.sfa, x.sfb, x.gsa, x.gsb, workspace)
    elif w.fp4 and w.unaligned:
        kgw.kgw_wgrad_fp4_unaligned(args, x.sfa, x.sfb, workspace)
    elif w.fp8 and w.unaligned:
        kgw.kgw_wgrad_fp8_unaligned(args, x.sfa, x.sfb, 1 if w.sf_format == "ue8m0_32" else 0, workspace)
    elif w.fp4:
        kgw.kgw_wgrad_fp4_ue8m0(args, x.sfa, x.sfb, workspace)
    elif w.fp8 and w.sf_format == "ue8m0_32":
        kgw.kgw_wgrad_fp8_ue8m0(args, x.sfa, x.sfb, workspace)
    elif w.fp8:
        kgw.kgw_wgrad_fp8_blockscaled(args, x.sfa, x.sfb, workspace)
    elif w.unaligned:
        kgw.kgw_wgrad_bf16_unaligned(args, workspace)
    else:
        kgw.kgw_wgrad_bf16(args, workspace)
    return outs


def oracle_full(w, x_cpu):
    import oracle.kgw_oracle as O
    dec_bits = bits8 if (w.fp8 or w.fp4) else bits16
    c = None if x_cpu.c is None else to_f64(x_cpu.c)
    return O.wgrad_from_storage(dec_bits(x_cpu.a), dec_bits(x_cpu.b), x_cpu.offsets.numpy(), w.hidden,
                                w.intermediate, input_order=w.input_order, fp8=w.fp8,
                                sfa=None if x_cpu.sfa is None else x_cpu.sfa.numpy(),
                                sfb=None if x_cpu.sfb is None else x_cpu.sfb.numpy(),
                                c_init=c, accumulate=w.accumulate, a_major=w.a_major, b_major=w.b_major,
                                sf_format=w.sf_format, fp4=w.fp4,
                                global_scale_a=None if x_cpu.gsa is None else float(x_cpu.gsa[0]),
                                global_scale_b=None if x_cpu.gsb is None else float(x_cpu.gsb[0]))


def assert_close_to_oracle(w, got: np.ndarray, ref: np.ndarray, S: np.ndarray, c_init=None):
    import oracle.kgw_oracle as O
    tol = O.tolerance(S, ref, w.out_dtype, c_init if (w.accumulate and w.out_dtype == "f32") else None)
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:8]
        msg = "; ".join(f"{tuple(i)} got={got[tuple(i)]:.6g} ref={ref[tuple(i)]:.6g} tol={tol[tuple(i)]:.3g}"
                        for i in idx)
        raise AssertionError(f"{int(bad.sum())} of {bad.size} elements out of tolerance: {msg}")


def check_full(w, label=None, device="cuda"):
    """Run workload ``w`` on the GPU and compare every output element with the oracle."""
    import oracle.kgw_oracle as O
    import workloads as W
    kgw = ensure_built()
    x_cpu = W.make_inputs(w, "cpu")
    x = W.Inputs(*[None if t is None else t.to(device) for t in
                   (x_cpu.a, x_cpu.b, x_cpu.offsets, x_cpu.sfa, x_cpu.sfb, x_cpu.c, x_cpu.gsa, x_cpu.gsb)])
    status = torch.full((1,), -1, dtype=torch.int32, device=device)
    outs = run_gpu(w, x, device, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact()
    bits = bits8 if (w.fp8 or w.fp4) else bits16
    a_bits, b_bits = bits(x_cpu.a), bits(x_cpu.b)
    offsets = x_cpu.offsets.numpy()
    sf = dict(sfa=None if x_cpu.sfa is None else x_cpu.sfa.numpy(),
              sfb=None if x_cpu.sfb is None else x_cpu.sfb.numpy(),
              global_scale_a=None if x_cpu.gsa is None else float(x_cpu.gsa[0]),
              global_scale_b=None if x_cpu.gsb is None else float(x_cpu.gsb[0]))
    counts = np.asarray(w.counts)
    worst, checked, bad = 0.0, 0, []
    for e in range(w.num_experts):
        if counts[e] == 0:
            if w.accumulate:
                assert torch.equal(outs.views[e], x.c[e]), f"empty expert {e} changed"
            else:
                assert not outs.views[e].any(), f"empty expert {e} not zero"
            continue
        r, s = O.expert_from_storage(a_bits, b_bits, offsets, w.hidden, w.intermediate, e,
                                     input_order=w.input_order, fp8=w.fp8, a_major=w.a_major, b_major=w.b_major,
                                     sf_format=w.sf_format, fp4=w.fp4, **sf)
        c = to_f64(x_cpu.c[e]) if w.accumulate else None
        ref = r if c is None else c + r
        tol = O.tolerance(s, ref, w.out_dtype, c if (w.accumulate and w.out_dtype == "f32") else None)
        got = to_f64(outs.views[e])
        err = np.abs(got - ref)
        ratio = err / tol
        worst = max(worst, float(np.nanmax(ratio)) if ratio.size else 0.0)
        checked += ref.size
        over = ~(err <= tol)
        if over.any():
            i = tuple(np.argwhere(over)[0])
            bad.append((e, int(over.sum()), i, float(got[i]), float(ref[i]), float(tol[i])))
    print(f"[full parity] {label or w.name}: {checked} elements, worst err/tol = {worst:.3g}")
    assert not bad, f"experts out of tolerance (expert, count, first index, got, ref, tol): {bad[:5]}"
    return worst
