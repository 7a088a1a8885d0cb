"""Parity of the M-grouped GEMM (kgw_mgrouped_bf16) with the CPU oracle, through the C ABI.

Small cases (several tiles, empty groups, unsorted index blocks, masked groups with partial
tiles and max_m not a multiple of 128, every output type, accumulate) are compared with the full
oracle element by element; the full-size forward, dgrad and masked-decode workloads on sampled
rows. Tolerance per element: |gpu - oracle| <= 2e-5*S + 1e-6 with S = |A_r| @ |op(B_g)| (FP32
accumulation over K), plus one rounding to the output type (2**-8|ref| BF16, 2**-10|ref| + 2**-24
FP16) and, when accumulating into FP32, 2**-23(|C| + |ref|). Rows that no group owns must keep
their previous contents bit for bit, and nothing outside D may change.
"""
import numpy as np
import pytest
import torch

import oracle.kgw_oracle as KO
import oracle.mgrouped_oracle as MO
import workloads.mgrouped as MW
from kgw_testlib import bits16, ensure_built, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096
CANARY = 7.25


class MGOut:
    """D inside a guard band. Rows not written by the call hold d0 (masked/accumulate) or a canary."""

    def __init__(self, w, d0, rows=None):
        dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.out_dtype]
        rows = w.rows if rows is None else rows
        self.numel = rows * w.n
        self.buf = torch.full((self.numel + 2 * GUARD,), CANARY, dtype=dt, device=DEV)
        self.d = self.buf[GUARD:GUARD + self.numel].view(rows, w.n)
        if d0 is not None:
            self.d.copy_(d0.reshape(rows, w.n))

    def guards_intact(self):
        return bool(torch.all(self.buf[:GUARD] == CANARY) and torch.all(self.buf[-GUARD:] == CANARY))


def run_mg(w, x, out, status=None, workspace=None):
    kgw = ensure_built()
    lay = {"offsets": kgw.KGW_MG_OFFSETS, "indices": kgw.KGW_MG_INDICES, "masked": kgw.KGW_MG_MASKED}[w.layout]
    odt = {"f32": kgw.KGW_OUT_F32, "bf16": kgw.KGW_OUT_BF16, "f16": kgw.KGW_OUT_F16}[w.out_dtype]
    args = kgw.make_mgrouped_args(w.num_groups, w.m, w.n, w.k, x.a, x.b, x.groups, out.d, layout=lay,
                                  b_major=kgw.KGW_K_MAJOR if w.b_major == "k" else kgw.KGW_MN_MAJOR,
                                  out_dtype=odt, accumulate=w.accumulate, status_dev=status)
    if workspace is None:
        workspace = torch.empty(kgw.kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=DEV)
    if w.fp8:
        kgw.kgw_mgrouped_fp8(args, x.sfa, x.sfb, 1 if w.sf_format == "ue8m0_32" else 0, workspace)
    else:
        kgw.kgw_mgrouped_bf16(args, workspace)
    return args


def u8(t):
    return t.contiguous().view(torch.uint8).numpy()


def oracle_ref(w, x_cpu):
    d0 = None if x_cpu.d0 is None else to_f64(x_cpu.d0).reshape(w.rows, w.n)
    if w.fp8:
        return MO.mgrouped_fp8_from_storage(u8(x_cpu.a), u8(x_cpu.b), x_cpu.sfa.numpy(), x_cpu.sfb.numpy(),
                                            w.layout, x_cpu.groups.numpy(), w.m, b_major=w.b_major,
                                            sf_format=w.sf_format, d_init=d0, accumulate=w.accumulate)
    return MO.mgrouped_from_storage(bits16(x_cpu.a), bits16(x_cpu.b), w.layout, x_cpu.groups.numpy(), w.m,
                                    b_major=w.b_major, d_init=d0, accumulate=w.accumulate)


def check_close(w, got, ref, S, c=None):
    tol = KO.tolerance(S, ref, w.out_dtype, c if (w.accumulate and w.out_dtype == "f32") else None)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        msg = "; ".join(f"{tuple(i)} got={got[tuple(i)]:.6g} ref={ref[tuple(i)]:.6g} tol={tol[tuple(i)]:.3g}"
                        for i in idx)
        raise AssertionError(f"{int(bad.sum())} of {bad.size} elements out of tolerance: {msg}")


def _check(w):
    kgw = ensure_built()
    x_cpu = MW.make_mg_inputs(w, "cpu")
    x = MW.make_mg_inputs(w, DEV)
    out = MGOut(w, x.d0)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    run_mg(w, x, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert out.guards_intact(), "write outside D"
    got = to_f64(out.d)
    ref, S = oracle_ref(w, x_cpu)
    own = MO.owned_mask(w.layout, x_cpu.groups.numpy(), w.m, w.num_groups, w.rows)
    c = None if x_cpu.d0 is None else to_f64(x_cpu.d0).reshape(w.rows, w.n)
    check_close(w, got[own], ref[own], S[own], None if c is None else c[own])
    if (~own).any():
        before = x_cpu.d0.reshape(w.rows, w.n)[torch.from_numpy(~own)]
        assert torch.equal(out.d.cpu()[torch.from_numpy(~own)], before), "rows owned by no group changed"
    return out


C = MW.mg_custom
CASES = {
    "tiny": MW.mg_tiny(),
    "offsets_forward_bf16": C(4, 512, 256, "offsets", [256, 0, 384, 128], seed=41),
    "offsets_dgrad_bf16": C(4, 512, 256, "offsets", [256, 0, 384, 128], seed=42, b_major="mn"),
    "offsets_f32_long_k": C(3, 256, 1024, "offsets", [128, 512, 256], seed=43, out_dtype="f32"),
    "offsets_f16": C(3, 768, 192, "offsets", [384, 128, 0], seed=44, out_dtype="f16"),
    "offsets_accumulate_f32": C(3, 256, 320, "offsets", [256, 256, 128], seed=45, out_dtype="f32",
                                accumulate=True),
    "offsets_accumulate_bf16_dgrad": C(2, 512, 128, "offsets", [128, 384], seed=46, accumulate=True,
                                       b_major="mn"),
    "indices_sorted": C(4, 256, 128, "indices", [128, 256, 0, 128], seed=47),
    "indices_shuffled": C(5, 512, 192, "indices", [384, 128, 0, 256, 128], seed=48, shuffle_blocks=True),
    "indices_shuffled_dgrad_f32": C(3, 256, 256, "indices", [256, 128, 384], seed=49, shuffle_blocks=True,
                                    b_major="mn", out_dtype="f32"),
    "masked_partial_tiles": C(5, 512, 128, "masked", [1, 127, 129, 0, 256], seed=50, max_m=256),
    "masked_odd_max_m": C(4, 256, 256, "masked", [200, 0, 73, 131], seed=51, max_m=200),
    "masked_accumulate_f32_dgrad": C(3, 256, 192, "masked", [64, 300, 0], seed=52, max_m=320,
                                     out_dtype="f32", accumulate=True, b_major="mn"),
    "masked_all_empty": C(3, 256, 64, "masked", [0, 0, 0], seed=53, max_m=128),
    "many_groups": C(40, 256, 128, "offsets", [128 * (i % 3) for i in range(40)], seed=54),
    # FP8 (e4m3 with per-128-K scales per row of A and per column of each weight)
    "fp8_offsets_forward": C(4, 512, 256, "offsets", [256, 0, 384, 128], seed=70, fp8=True, b_std=1.0),
    "fp8_dgrad_f32": C(3, 256, 512, "offsets", [128, 256, 128], seed=71, fp8=True, b_std=1.0, b_major="mn",
                       out_dtype="f32"),
    "fp8_indices_shuffled_ue8m0": C(4, 256, 256, "indices", [256, 128, 0, 256], seed=72, fp8=True, b_std=1.0,
                                    shuffle_blocks=True, sf_format="ue8m0_32"),
    "fp8_masked_partial_tiles": C(4, 512, 384, "masked", [1, 129, 0, 200], seed=73, fp8=True, b_std=1.0, max_m=256),
    "fp8_masked_accumulate_f16": C(3, 256, 256, "masked", [64, 300, 17], seed=74, fp8=True, b_std=1.0, max_m=320,
                                   accumulate=True, out_dtype="f16"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_mgrouped_parity_small(name):
    _check(CASES[name])


def test_offsets_indices_same_result():
    """The same rows grouped by offsets and by per-row ids give bit-identical D."""
    kgw = ensure_built()
    w1 = C(3, 512, 256, "offsets", [256, 0, 384], seed=60)
    w2 = C(3, 512, 256, "indices", [256, 0, 384], seed=60)
    x1 = MW.make_mg_inputs(w1, DEV)
    x2 = MW.make_mg_inputs(w2, DEV)
    assert torch.equal(x1.a, x2.a) and torch.equal(x1.b, x2.b)
    o1, o2 = MGOut(w1, None), MGOut(w2, None)
    run_mg(w1, x1, o1)
    run_mg(w2, x2, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1.d, o2.d)


def test_dgrad_equals_forward_of_transposed_weight():
    """op(B) = B for N-major storage: D matches the K-major call on the transposed weights."""
    w1 = C(2, 256, 128, "offsets", [256, 128], seed=61, b_major="mn")
    x = MW.make_mg_inputs(w1, DEV)
    w2 = C(2, 256, 128, "offsets", [256, 128], seed=61, b_major="k")
    x2 = MW.MGInputs(x.a, x.b.transpose(1, 2).contiguous(), x.groups, None)
    o1, o2 = MGOut(w1, None), MGOut(w2, None)
    run_mg(w1, x, o1)
    run_mg(w2, x2, o2)
    torch.cuda.synchronize()
    # same products, possibly different MMA summation order inside a K step: compare to each other
    a = to_f64(o1.d)
    b = to_f64(o2.d)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 1e-3)


def test_deterministic():
    w = C(4, 512, 512, "offsets", [512, 128, 0, 256], seed=62, out_dtype="f32")
    x = MW.make_mg_inputs(w, DEV)
    o1, o2 = MGOut(w, None), MGOut(w, None)
    run_mg(w, x, o1)
    run_mg(w, x, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1.d, o2.d)


@pytest.mark.parametrize("layout,groups,m", [
    ("offsets", [128, 200, 384], 384),          # count not a multiple of 128
    ("offsets", [256, 128, 384], 384),          # decreasing
    ("offsets", [128, 256, 256], 384),          # last != m
    ("indices", None, 384),                     # a 128-row block with two ids
    ("indices", [5] * 384, 384),                # id out of range
    ("masked", [10, 129, 3], 128),              # masked_m > max_m
    ("masked", [10, -1, 3], 128),               # negative
])
def test_device_detected_layout_errors(layout, groups, m):
    """Invalid group descriptions set KGW_ERR_OFFSETS on the device and leave D untouched."""
    kgw = ensure_built()
    G, N, K = 3, 256, 64
    if groups is None:
        groups = np.repeat([0, 1, 2], 128)
        groups[129] = 2
    rows = G * m if layout == "masked" else m
    w = C(G, N, K, layout, [0] * G, seed=63, max_m=m if layout == "masked" else 0)
    a = torch.randn(rows, K, device=DEV).to(torch.bfloat16)
    b = torch.randn(G, N, K, device=DEV).to(torch.bfloat16)
    g = torch.tensor(np.asarray(groups, dtype=np.int32), device=DEV)
    out = MGOut(w, None, rows=rows)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    lay = {"offsets": kgw.KGW_MG_OFFSETS, "indices": kgw.KGW_MG_INDICES, "masked": kgw.KGW_MG_MASKED}[layout]
    args = kgw.make_mgrouped_args(G, m, N, K, a, b, g, out.d, layout=lay, status_dev=status)
    ws = torch.empty(kgw.kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=DEV)
    kgw.kgw_mgrouped_bf16(args, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_ERR_OFFSETS
    assert torch.all(out.buf == CANARY), "an invalid call wrote output"


def test_host_detected_errors():
    kgw = ensure_built()
    a = torch.zeros(256, 128, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(2, 256, 128, dtype=torch.bfloat16, device=DEV)
    g = torch.tensor([128, 256], dtype=torch.int32, device=DEV)
    d = torch.zeros(256, 256, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    mk = kgw.make_mgrouped_args

    def rc(args, nbytes=None):
        return kgw.kgw_mgrouped_bf16(args, ws, workspace_bytes=nbytes, check=False)

    assert rc(mk(2, 256, 256, 128, a, b, g, d)) == kgw.KGW_OK
    assert rc(mk(2, 256, 128, 128, a, b, g, d)) == kgw.KGW_ERR_UNSUPPORTED        # n % 256
    assert rc(mk(2, 256, 256, 96, a, b, g, d)) == kgw.KGW_ERR_UNSUPPORTED         # k % 64
    assert rc(mk(2, 200, 256, 128, a, b, g, d)) == kgw.KGW_ERR_INVALID_ARG        # m % 128 (contiguous)
    assert rc(mk(0, 256, 256, 128, a, b, g, d)) == kgw.KGW_ERR_INVALID_ARG        # G = 0
    assert rc(mk(2, 256, 256, 128, a, b, g, d, layout=7)) == kgw.KGW_ERR_INVALID_ARG
    assert rc(mk(2, 256, 256, 128, a, b, g, d, out_dtype=9)) == kgw.KGW_ERR_INVALID_ARG
    assert rc(mk(2, 256, 256, 128, a, b, None, d)) == kgw.KGW_ERR_INVALID_ARG     # no group description
    assert rc(mk(2, 256, 256, 128, a.data_ptr() + 2, b, g, d)) == kgw.KGW_ERR_ALIGNMENT
    assert rc(mk(2, 256, 256, 128, a, b, g, d), nbytes=16) == kgw.KGW_ERR_WORKSPACE
    torch.cuda.synchronize()


def test_binding_convenience_call():
    kgw = ensure_built()
    w = C(3, 256, 128, "offsets", [128, 0, 256], seed=64)
    x_cpu = MW.make_mg_inputs(w, "cpu")
    x = MW.make_mg_inputs(w, DEV)
    d = kgw.mgrouped(x.a, x.b, x.groups)
    torch.cuda.synchronize()
    ref, S = oracle_ref(w, x_cpu)
    check_close(w, to_f64(d), ref, S)


def test_graph_capture_replays():
    """No host synchronisation: the call can be captured in a CUDA graph (section 2.2's reason
    for the masked layout) and replays with new masked_m values."""
    kgw = ensure_built()
    w = C(3, 256, 128, "masked", [5, 100, 0], seed=65, max_m=128)
    x = MW.make_mg_inputs(w, DEV)
    out = MGOut(w, x.d0)
    args = kgw.make_mgrouped_args(3, 128, 256, 128, x.a, x.b, x.groups, out.d, layout=kgw.KGW_MG_MASKED)
    ws = torch.empty(kgw.kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kgw.kgw_mgrouped_bf16(args, ws, stream=s)   # first call on this stream outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kgw.kgw_mgrouped_bf16(args, ws, stream=s)
    for mm in ([128, 0, 17], [1, 2, 3]):
        x.groups.copy_(torch.tensor(mm, dtype=torch.int32))
        out.d.copy_(x.d0.reshape(w.rows, w.n))
        g.replay()
        torch.cuda.synchronize()
        w2 = C(3, 256, 128, "masked", mm, seed=65, max_m=128)
        x_cpu = MW.make_mg_inputs(w2, "cpu")
        ref, S = oracle_ref(w2, x_cpu)
        own = MO.owned_mask("masked", np.array(mm), 128, 3, w.rows)
        got = to_f64(out.d)
        check_close(w2, got[own], ref[own], S[own])
        assert torch.equal(out.d.cpu()[torch.from_numpy(~own)], x_cpu.d0.reshape(w.rows, w.n)[torch.from_numpy(~own)])


# ------------------------------------------------------------------------------------------
# Full-size workloads: every owned row against the oracle, unowned rows bit-exact
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["mg_forward", "mg_dgrad", "mg_masked", "mg_fp8_forward", "mg_fp8_masked"])
def test_mgrouped_full_size(name):
    kgw = ensure_built()
    w = MW.MG_NAMED[name]()
    x_cpu = MW.make_mg_inputs(w, "cpu")
    x = MW.MGInputs(x_cpu.a.to(DEV), x_cpu.b.to(DEV), x_cpu.groups.to(DEV),
                    None if x_cpu.d0 is None else x_cpu.d0.to(DEV),
                    None if x_cpu.sfa is None else x_cpu.sfa.to(DEV), None if x_cpu.sfb is None else x_cpu.sfb.to(DEV))
    out = MGOut(w, x.d0)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    run_mg(w, x, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert out.guards_intact()
    own = MO.owned_mask(w.layout, x_cpu.groups.numpy(), w.m, w.num_groups, w.rows)
    ref, S = oracle_ref(w, x_cpu)
    got = to_f64(out.d)
    c = None if x_cpu.d0 is None else to_f64(x_cpu.d0).reshape(w.rows, w.n)
    tol = KO.tolerance(S[own], ref[own], w.out_dtype,
                       c[own] if (c is not None and w.accumulate and w.out_dtype == "f32") else None)
    print(f"[full parity] {name}: {int(own.sum()) * w.n} elements, worst err/tol = "
          f"{float(np.max(np.abs(got[own] - ref[own]) / tol)):.3g}")
    check_close(w, got[own], ref[own], S[own], None if c is None else c[own])
    if (~own).any():
        mask = torch.from_numpy(~own).to(DEV)
        assert torch.equal(out.d[mask], x.d0.reshape(w.rows, w.n)[mask]), "rows past masked_m changed"


def test_fp8_host_rules():
    """FP8: k must be a multiple of 128; scales must be given and 16-byte aligned."""
    kgw = ensure_built()
    a = torch.zeros(256, 192, dtype=torch.uint8, device=DEV)
    b = torch.zeros(2, 256, 192, dtype=torch.uint8, device=DEV)
    g = torch.tensor([128, 256], dtype=torch.int32, device=DEV)
    d = torch.zeros(256, 256, dtype=torch.bfloat16, device=DEV)
    sf = torch.ones(8 * 256, dtype=torch.float32, device=DEV)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    args = kgw.make_mgrouped_args(2, 256, 256, 192, a, b, g, d)
    assert kgw.kgw_mgrouped_fp8(args, sf, sf, 0, ws, check=False) == kgw.KGW_ERR_UNSUPPORTED       # k % 128
    args = kgw.make_mgrouped_args(2, 256, 256, 128, a, b, g, d)
    assert kgw.kgw_mgrouped_fp8(args, None, sf, 0, ws, check=False) == kgw.KGW_ERR_INVALID_ARG
    assert kgw.kgw_mgrouped_fp8(args, sf.data_ptr() + 4, sf, 0, ws, check=False) == kgw.KGW_ERR_ALIGNMENT
    assert kgw.kgw_mgrouped_fp8(args, sf, sf, 5, ws, check=False) == kgw.KGW_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["offsets_forward_bf16", "indices_shuffled", "masked_partial_tiles",
                                  "masked_odd_max_m", "offsets_accumulate_bf16_dgrad"])
def test_single_cta_and_pair_rows_agree(name):
    """BF16 calls run on CTA pairs (two 128-row tiles of one group per work row; a group with an
    odd tile count ends with a half-empty row). The same call on single-CTA tiles gives the same
    bits, and rows outside the groups stay untouched either way."""
    kgw = ensure_built()
    w = CASES[name]
    x = MW.make_mg_inputs(w, DEV)
    o_pair = MGOut(w, x.d0)
    run_mg(w, x, o_pair)
    prev = kgw.kgw_debug_set(3, 1)
    try:
        o_single = MGOut(w, x.d0)
        run_mg(w, x, o_single)
    finally:
        kgw.kgw_debug_set(3, prev)
    torch.cuda.synchronize()
    assert o_pair.guards_intact() and o_single.guards_intact()
    assert torch.equal(o_pair.buf.view(torch.int16) if o_pair.buf.element_size() == 2 else o_pair.buf,
                       o_single.buf.view(torch.int16) if o_single.buf.element_size() == 2 else o_single.buf)


@pytest.mark.parametrize("layout", ["offsets", "indices", "masked"])
def test_no_rows_at_all(layout):
    """A call with no rows (every group empty) enqueues nothing harmful and reports KGW_OK."""
    kgw = ensure_built()
    G = 3
    b = torch.zeros(G, 256, 64, dtype=torch.bfloat16, device=DEV)
    groups = torch.zeros(G, dtype=torch.int32, device=DEV)
    m = 128 if layout == "masked" else 0
    a = torch.zeros(max(1, G * m), 64, dtype=torch.bfloat16, device=DEV)
    d = torch.full((max(1, G * m), 256), 7.25, dtype=torch.bfloat16, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    lay = {"offsets": kgw.KGW_MG_OFFSETS, "indices": kgw.KGW_MG_INDICES, "masked": kgw.KGW_MG_MASKED}[layout]
    args = kgw.make_mgrouped_args(G, m, 256, 64, a if m else None, b, groups if layout != "indices" else None,
                                  d if m else None, layout=lay, status_dev=status)
    ws = torch.empty(kgw.kgw_mgrouped_workspace_size(args), dtype=torch.uint8, device=DEV)
    kgw.kgw_mgrouped_bf16(args, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_OK
    assert torch.all(d == 7.25)
