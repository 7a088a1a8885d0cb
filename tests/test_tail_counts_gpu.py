"""Token counts that are not multiples of 256 (kgw_wgrad_bf16_unaligned).

First the per-expert descriptors that the schedule kernel builds for the token tails (the
operand's own descriptor with the token extent cut at the expert's last token) are compared
byte for byte with host encodings; only the schedule kernel runs there. The parity cases after
it use those descriptors for copies and are skipped if any descriptor differed. Parity follows
the other parity tests: every element against the float64 oracle within
2e-5*S + 1e-6 (+ one output rounding), empty experts exact, nothing written outside the outputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from kgw_testlib import Outputs, assert_close_to_oracle, ensure_built, oracle_full, run_gpu, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
_MAPS_OK = {"checked": False, "ok": True}

MAJORS = [("k", "mn"), ("mn", "mn"), ("k", "k"), ("mn", "k")]


def _map_check(counts, H, I, a_major, b_major, order):
    kgw = ensure_built()
    counts = np.asarray(counts, dtype=np.int64)
    T = int(counts.sum())
    offsets = np.cumsum(counts).astype(np.int32)
    a = torch.empty(H * T, dtype=torch.bfloat16, device=DEV)
    b = torch.empty(I * T, dtype=torch.bfloat16, device=DEV)
    off_d = torch.from_numpy(offsets).to(DEV)
    out = torch.empty((len(counts), H, I), dtype=torch.float32, device=DEV)
    args = kgw.make_args(len(counts), H, I, T, a, b, off_d, out=out,
                         input_order=kgw.KGW_RAGGED if order == "ragged" else kgw.KGW_TENSOR2D,
                         a_major=kgw.KGW_MN_MAJOR if a_major == "mn" else kgw.KGW_K_MAJOR,
                         b_major=kgw.KGW_K_MAJOR if b_major == "k" else kgw.KGW_MN_MAJOR)
    ws = kgw.workspace_for(args, device=DEV)
    dump = np.zeros(len(counts) * 512, dtype=np.uint8)
    mism = kgw.kgw_debug_check_tail_maps(args, offsets, ws, host_dump=dump)
    if mism != 0:
        _MAPS_OK["ok"] = False
        d = dump.reshape(len(counts), 2, 2, 128)
        msgs = []
        for e in np.nonzero(counts)[0]:
            for op in range(2):
                diff = np.nonzero(d[e, op, 0] != d[e, op, 1])[0]
                if len(diff):
                    msgs.append(f"expert {e} operand {'AB'[op]} (end={offsets[e]}) bytes {diff.tolist()}")
        pytest.fail(f"{mism} descriptors differ; " + "; ".join(msgs[:4]))


@pytest.mark.parametrize("a_major,b_major", MAJORS)
@pytest.mark.parametrize("counts,H,I", [
    ([8, 0, 72, 1000], 128, 256),                         # small: token extents x row bytes < 128 KiB
    ([264, 1208, 0, 56, 4096], 512, 512),
    ([4128, 5200, 3224, 5200, 3632, 3904, 4904, 3872], 4096, 2048),
])
def test_tail_descriptors_match_host_encoding(counts, H, I, a_major, b_major):
    _MAPS_OK["checked"] = True
    _map_check(counts, H, I, a_major, b_major, "tensor2d")


@pytest.mark.parametrize("a_major,b_major", MAJORS)
def test_tail_descriptors_ragged_order(a_major, b_major):
    _MAPS_OK["checked"] = True
    _map_check([24, 1000, 0, 136], 256, 512, a_major, b_major, "ragged")


def _require_maps():
    if not _MAPS_OK["checked"] or not _MAPS_OK["ok"]:
        pytest.skip("token-tail descriptors were not verified against host encodings")


def _check(w):
    _require_maps()
    kgw = ensure_built()
    x_cpu = W.make_inputs(w, "cpu")
    x = W.make_inputs(w, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact(), "write outside the output buffers"
    got = to_f64(outs.stacked())
    ref, S = oracle_full(w, x_cpu)
    c = None if x_cpu.c is None else to_f64(x_cpu.c)
    assert_close_to_oracle(w, got, ref, S, c)
    for e in np.nonzero(np.asarray(w.counts) == 0)[0]:
        if w.accumulate:
            assert torch.equal(outs.views[e].cpu(), x_cpu.c[e])
        else:
            assert not outs.views[e].any()


def U(*args, **kw):
    return W.custom(*args, unaligned=True, **kw)


CASES = {
    "k_major_a_single": U(4, 384, 512, [8, 0, 72, 1000], seed=120),
    "pair_tails": U(5, 512, 512, [264, 1208, 0, 56, 4096], seed=121),
    "both_mn_major_any_count": U(5, 256, 512, [1, 7, 130, 0, 999], seed=122, a_major="mn"),
    "k_major_b_bf16": U(3, 256, 768, [40, 200, 8], seed=123, b_major="k", out_dtype="bf16"),
    "ragged_k_major_a": U(4, 256, 512, [24, 1000, 0, 136], seed=124, input_order="ragged"),
    "ragged_mn_a_k_b": U(3, 384, 256, [88, 0, 1304], seed=125, input_order="ragged", a_major="mn", b_major="k"),
    "split_k_tail": U(2, 256, 256, [10008, 8], seed=126),
    "pair_split_k_tail_accumulate": U(3, 512, 256, [12296, 0, 520], seed=127, accumulate=True, out_dtype="bf16"),
    "discrete_f16": U(3, 256, 512, [136, 8, 2000], seed=128, output_mode="discrete", out_dtype="f16"),
    "aligned_counts_same_as_bf16": U(3, 256, 512, [256, 0, 768], seed=129),
}


@pytest.mark.parametrize("name", list(CASES))
def test_tail_parity_small(name):
    _check(CASES[name])


def test_aligned_counts_bitwise_equal_the_pages_entry():
    """With counts that are multiples of 256 the unaligned entry computes what kgw_wgrad_bf16 does."""
    _require_maps()
    w = W.custom(3, 512, 512, [768, 0, 1280], seed=130)
    x = W.make_inputs(w, DEV)
    a = run_gpu(w, x, DEV).stacked().clone()
    b = run_gpu(dataclasses.replace(w, unaligned=True), x, DEV).stacked().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("a_major,b_major,counts", [
    ("k", "mn", [4, 12, 64]),     # 4 and 12 are not multiples of 8 (K-major A); the total 80 is
    ("mn", "k", [16, 4, 12]),     # K-major B; the total 32 is
    ("k", "mn", [256, -8, 8]),    # negative
])
def test_device_rejects_counts_breaking_the_rule(a_major, b_major, counts):
    """A count that breaks the rule: KGW_ERR_OFFSETS on the device and no output written."""
    kgw = ensure_built()
    T = int(np.sum(np.abs(counts)))
    offs = np.cumsum(counts).astype(np.int32)
    w = W.custom(3, 128, 256, [0, 0, 0], seed=131, a_major=a_major, b_major=b_major, unaligned=True)
    outs = Outputs(w, DEV)
    a = torch.zeros(128 * T + 64, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(256 * T + 64, dtype=torch.bfloat16, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(3, 128, 256, int(offs[-1]), a, b, torch.from_numpy(offs).to(DEV), out=outs.dense,
                         a_major=kgw.KGW_MN_MAJOR if a_major == "mn" else kgw.KGW_K_MAJOR,
                         b_major=kgw.KGW_K_MAJOR if b_major == "k" else kgw.KGW_MN_MAJOR, status_dev=status)
    ws = kgw.workspace_for(args, device=DEV)
    kgw.kgw_wgrad_bf16_unaligned(args, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_ERR_OFFSETS
    assert torch.all(outs.buf == 7.25)


def test_full_unaligned():
    """The unaligned workload (balanced shape, counts multiples of 8) at full size, every element."""
    _require_maps()
    from kgw_testlib import check_full
    check_full(W.unaligned(), "unaligned")


# ------------------------------------------------------------------------------------------
# Block-scaled entries with counts that are not multiples of 256 (kgw_wgrad_fp8_unaligned,
# kgw_wgrad_fp4_unaligned): scale blocks per expert, rows sum over f < e of ceil(n_f/128) on
# ------------------------------------------------------------------------------------------

_MAPS_BS = {"checked": False, "ok": True}


def _map_check_kind(kind, counts, H, I, a_major, b_major, order):
    kgw = ensure_built()
    counts = np.asarray(counts, dtype=np.int64)
    T = int(counts.sum())
    offsets = np.cumsum(counts).astype(np.int32)
    nbytes = T // 2 if kind == 2 else T
    a = torch.empty(max(1, H * nbytes), dtype=torch.uint8, device=DEV)
    b = torch.empty(max(1, I * nbytes), dtype=torch.uint8, device=DEV)
    off_d = torch.from_numpy(offsets).to(DEV)
    out = torch.empty((len(counts), H, I), dtype=torch.float32, device=DEV)
    args = kgw.make_args(len(counts), H, I, T, a, b, off_d, out=out,
                         input_order=kgw.KGW_RAGGED if order == "ragged" else kgw.KGW_TENSOR2D,
                         a_major=kgw.KGW_MN_MAJOR if a_major == "mn" else kgw.KGW_K_MAJOR,
                         b_major=kgw.KGW_K_MAJOR if b_major == "k" else kgw.KGW_MN_MAJOR)
    ws = kgw.workspace_for(args, True, device=DEV)
    dump = np.zeros(len(counts) * 512, dtype=np.uint8)
    mism = kgw.kgw_debug_check_tail_maps_kind(args, kind, offsets, ws, host_dump=dump)
    if mism != 0:
        _MAPS_BS["ok"] = False
        pytest.fail(f"{mism} descriptors differ from host encodings (kind {kind})")


@pytest.mark.parametrize("a_major,b_major", MAJORS)
@pytest.mark.parametrize("order", ["tensor2d", "ragged"])
def test_fp8_tail_descriptors_match_host_encoding(a_major, b_major, order):
    _MAPS_BS["checked"] = True
    _map_check_kind(1, [16, 0, 144, 1008, 4096], 256, 512, a_major, b_major, order)
    _map_check_kind(1, [4112, 5200, 3216, 5200], 4096, 1536, a_major, b_major, order)


@pytest.mark.parametrize("order", ["tensor2d", "ragged"])
def test_fp4_tail_descriptors_match_host_encoding(order):
    _MAPS_BS["checked"] = True
    _map_check_kind(2, [32, 0, 160, 1024, 4064], 256, 512, "k", "k", order)
    _map_check_kind(2, [4128, 5216, 3200, 5184], 4096, 1536, "k", "k", order)


def _require_bs_maps():
    if not _MAPS_BS["checked"] or not _MAPS_BS["ok"]:
        pytest.skip("block-scaled token-tail descriptors were not verified against host encodings")


def F8(*args, **kw):
    return W.custom(*args, unaligned=True, fp8=True, out_dtype=kw.pop("out_dtype", "f32"), **kw)


def F4(*args, **kw):
    return W.custom(*args, unaligned=True, fp4=True, b_major="k", sf_format="ue8m0_32", **kw)


BS_CASES = {
    "fp8_k_a_mn_b": F8(4, 256, 512, [16, 0, 144, 1008], seed=140),
    "fp8_ue8m0": F8(4, 256, 512, [48, 400, 0, 112], seed=141, sf_format="ue8m0_32"),
    "fp8_both_mn_any_count": F8(4, 128, 256, [1, 77, 0, 300], seed=142, a_major="mn"),
    "fp8_k_b": F8(3, 128, 768, [32, 208, 16], seed=143, b_major="k", out_dtype="bf16"),
    "fp8_ragged": F8(4, 256, 512, [96, 1040, 0, 16], seed=144, input_order="ragged"),
    "fp8_ragged_mn_a_k_b_ue8m0": F8(3, 384, 256, [80, 0, 1296], seed=145, input_order="ragged", a_major="mn",
                                    b_major="k", sf_format="ue8m0_32"),
    "fp8_split_k": F8(2, 128, 256, [12304, 16], seed=146),
    "fp8_split_k_accumulate": F8(3, 256, 256, [10000, 0, 528], seed=147, accumulate=True, out_dtype="bf16"),
    "fp8_discrete_f16": F8(3, 128, 512, [144, 16, 2000], seed=148, output_mode="discrete", out_dtype="f16"),
    "fp8_general_scales": F8(4, 256, 512, [48, 0, 1040, 16], seed=149, sf_format="f32_any", out_dtype="bf16"),
    "fp4": F4(4, 256, 512, [32, 0, 160, 1056], seed=150),
    "fp4_single_block_last_stage": F4(3, 128, 256, [96, 352, 128], seed=151, out_dtype="bf16"),
    "fp4_split_k": F4(2, 128, 256, [20000, 32], seed=152),
    "fp4_ragged": F4(4, 256, 512, [96, 0, 1184, 32], seed=155, input_order="ragged", out_dtype="bf16"),
}


@pytest.mark.parametrize("name", list(BS_CASES))
def test_block_scaled_tail_parity_small(name):
    _require_bs_maps()
    w = BS_CASES[name]
    from kgw_testlib import check_full
    check_full(w, name)


@pytest.mark.parametrize("fp4", [False, True])
def test_block_scaled_aligned_counts_bitwise_equal_the_pages_entries(fp4):
    """With counts that are multiples of 256 the unaligned block-scaled entries compute what the
    aligned ones do, bit for bit (the scale rows coincide)."""
    _require_bs_maps()
    kw = dict(fp4=True, b_major="k", sf_format="ue8m0_32") if fp4 else dict(fp8=True)
    w = W.custom(3, 256, 512, [768, 0, 1280], seed=153, **kw)
    x = W.make_inputs(w, DEV)
    a = run_gpu(w, x, DEV).stacked().clone()
    b = run_gpu(dataclasses.replace(w, unaligned=True), x, DEV).stacked().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("kind,counts", [(1, [16, 8, 40]), (2, [32, 16, 48]), (1, [32, -16, 16])])
def test_block_scaled_device_rejects_counts_breaking_the_rule(kind, counts):
    """FP8 with a K-major operand needs multiples of 16, FP4 multiples of 32: KGW_ERR_OFFSETS, nothing written."""
    kgw = ensure_built()
    T = int(np.sum(np.abs(counts)))
    offs = np.cumsum(counts).astype(np.int32)
    w = W.custom(3, 128, 256, [0, 0, 0], seed=154, unaligned=True)
    outs = Outputs(w, DEV)
    a = torch.zeros(128 * T + 64, dtype=torch.uint8, device=DEV)
    b = torch.zeros(256 * T + 64, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(8 * 256, dtype=torch.int32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(3, 128, 256, int(offs[-1]), a, b, torch.from_numpy(offs).to(DEV), out=outs.dense,
                         b_major=kgw.KGW_K_MAJOR if kind == 2 else kgw.KGW_MN_MAJOR, status_dev=status)
    ws = kgw.workspace_for(args, True, device=DEV)
    if kind == 1:
        kgw.kgw_wgrad_fp8_unaligned(args, sf, sf, 1, ws)
    else:
        kgw.kgw_wgrad_fp4_unaligned(args, sf, sf, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_ERR_OFFSETS
    assert torch.all(outs.buf == 7.25)


def test_full_fp8_unaligned():
    _require_bs_maps()
    from kgw_testlib import check_full
    check_full(W.fp8_unaligned(), "fp8 unaligned")
    check_full(dataclasses.replace(W.fp8_unaligned(), sf_format="ue8m0_32"), "fp8 unaligned ue8m0")


def test_full_fp4_unaligned():
    _require_bs_maps()
    from kgw_testlib import check_full
    check_full(W.fp4_unaligned(), "fp4 unaligned")
