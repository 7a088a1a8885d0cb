"""Parity of the CUDA path with the CPU oracle, element by element, through the C ABI.

Small cases span several 128x256 tiles, empty experts, split-K and both input orders and
output modes; the oracle evaluates them in full. Tolerance (per element, from the operation's
FP32 accumulation): |gpu - oracle| <= 2e-5*S + 1e-6 with S = |A_e| @ |B_e|, plus 2**-8*|ref|
for BF16 output (one final rounding) and 2**-23*(|C|+|ref|) when accumulating into FP32.
Empty experts must be exact (zeros, or the pre-filled output bit for bit).
"""
import numpy as np
import pytest
import torch

import workloads as W
from kgw_testlib import Outputs, assert_close_to_oracle, ensure_built, oracle_full, run_gpu, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _check(w, status_expected=0):
    kgw = ensure_built()
    x_cpu = W.make_inputs(w, "cpu")
    x = W.make_inputs(w, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == status_expected, kgw.kgw_status_string(int(status.item()))
    assert outs.guards_intact(), "write outside the output buffers"
    got = to_f64(outs.stacked())
    ref, S = oracle_full(w, x_cpu)
    c = None if x_cpu.c is None else to_f64(x_cpu.c)
    assert_close_to_oracle(w, got, ref, S, c)
    counts = np.asarray(w.counts)
    for e in np.nonzero(counts == 0)[0]:
        if w.accumulate:
            assert torch.equal(outs.views[e].cpu(), x_cpu.c[e]), f"empty expert {e} changed"
        else:
            assert not outs.views[e].any(), f"empty expert {e} not zero"
    return outs, got


CASES = {
    "tiny": W.tiny(),
    "multi_tile_f32": W.custom(5, 384, 768, [256, 0, 1280, 512, 2304], seed=21),
    "multi_tile_bf16": W.custom(5, 384, 768, [256, 0, 1280, 512, 2304], seed=22, out_dtype="bf16"),
    "accumulate_f32": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=23, accumulate=True),
    "accumulate_bf16": W.custom(4, 256, 512, [0, 512, 0, 256], seed=24, accumulate=True, out_dtype="bf16"),
    "ragged_f32": W.custom(5, 384, 512, [768, 256, 0, 1536, 512], seed=25, input_order="ragged"),
    "discrete_bf16": W.custom(4, 256, 768, [512, 0, 256, 1024], seed=26, out_dtype="bf16",
                              output_mode="discrete"),
    "ragged_discrete_accumulate": W.custom(3, 256, 512, [1024, 0, 768], seed=27, input_order="ragged",
                                           output_mode="discrete", accumulate=True, out_dtype="bf16"),
    "split_k": W.custom(2, 256, 512, [8192, 256], seed=28),
    "split_k_bf16_accumulate": W.custom(3, 128, 256, [6144, 0, 12288], seed=29, accumulate=True,
                                        out_dtype="bf16"),
    "split_k_ragged_discrete": W.custom(3, 256, 256, [256, 10240, 512], seed=30, input_order="ragged",
                                        output_mode="discrete", out_dtype="bf16"),
    "all_empty_overwrite": W.custom(3, 128, 256, [0, 0, 0], seed=31),
    "all_empty_accumulate": W.custom(3, 128, 256, [0, 0, 0], seed=32, accumulate=True),
    "single_expert": W.custom(1, 256, 512, [4096], seed=33, b_std=0.02),
    "many_experts": W.custom(256, 128, 256, np.random.default_rng(34).choice([0, 256, 512], 256), seed=34,
                             out_dtype="bf16"),
    # hidden a multiple of 256: BF16 tiles run on CTA pairs (256 x 256 per pair)
    "pair_multi_tile": W.custom(4, 768, 512, [1280, 0, 256, 2048], seed=64),
    "pair_bf16_accumulate_ragged": W.custom(3, 512, 768, [768, 256, 0], seed=65, accumulate=True,
                                            out_dtype="bf16", input_order="ragged"),
    "pair_split_k_discrete": W.custom(2, 512, 256, [16384, 256], seed=66, output_mode="discrete",
                                      out_dtype="bf16"),
    # operand storage orders: M-major A ([tokens, hidden]) and K-major B ([intermediate, tokens])
    "a_mn_pair": W.custom(4, 512, 512, [768, 0, 1280, 256], seed=90, a_major="mn"),
    "b_k_pair_bf16": W.custom(3, 512, 768, [1024, 256, 512], seed=91, b_major="k", out_dtype="bf16"),
    "a_mn_b_k_single_ragged": W.custom(4, 384, 512, [768, 256, 0, 2048], seed=92, a_major="mn", b_major="k",
                                       input_order="ragged"),
    "b_k_ragged_pair_split_accumulate": W.custom(2, 512, 256, [12288, 512], seed=93, b_major="k",
                                                 input_order="ragged", accumulate=True, out_dtype="bf16"),
    "fp8_a_mn": W.custom(3, 256, 512, [512, 768, 256], seed=94, fp8=True, a_major="mn", out_dtype="bf16"),
    "fp8_b_k_ragged": W.custom(3, 384, 512, [1280, 0, 512], seed=95, fp8=True, b_major="k", input_order="ragged"),
    "f16_out_pair": W.custom(4, 512, 512, [768, 0, 1024, 256], seed=97, out_dtype="f16"),
    "f16_accumulate_single_split": W.custom(3, 384, 256, [8192, 0, 512], seed=98, out_dtype="f16", accumulate=True),
    "fp8_f16_out": W.custom(2, 256, 512, [512, 1280], seed=99, fp8=True, out_dtype="f16"),
    "fp8_ue8m0_32": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=100, fp8=True, sf_format="ue8m0_32"),
    "fp8_ue8m0_32_ragged_mn_a": W.custom(3, 384, 512, [1280, 256, 0], seed=101, fp8=True, sf_format="ue8m0_32",
                                         input_order="ragged", a_major="mn", out_dtype="bf16"),
    "fp8_bf16_out": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=60, fp8=True, out_dtype="bf16"),
    "fp8_f32_ragged": W.custom(3, 384, 768, [256, 1280, 0], seed=61, fp8=True, input_order="ragged"),
    "fp8_split_k_accumulate": W.custom(3, 128, 256, [16384, 0, 256], seed=62, fp8=True, accumulate=True),
    "fp8_discrete": W.custom(3, 256, 256, [1024, 512, 256], seed=63, fp8=True, out_dtype="bf16",
                             output_mode="discrete"),
    "fp8_pair_ragged_split_k": W.custom(3, 512, 512, [16384, 0, 768], seed=68, fp8=True, input_order="ragged",
                                        out_dtype="bf16"),
    "fp8_single_cta_accumulate": W.custom(2, 384, 512, [1280, 512], seed=69, fp8=True, accumulate=True),
    # FP4 e2m1, K-major A and B, UE8M0 scales per 32 tokens (256 tokens per pipeline stage)
    "fp4_bf16_out": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=110, fp4=True, b_major="k",
                             sf_format="ue8m0_32", out_dtype="bf16"),
    "fp4_f32_multi_tile": W.custom(3, 384, 768, [256, 2048, 0], seed=111, fp4=True, b_major="k",
                                   sf_format="ue8m0_32"),
    "fp4_split_k_accumulate": W.custom(3, 128, 256, [32768, 0, 256], seed=112, fp4=True, b_major="k",
                                       sf_format="ue8m0_32", accumulate=True),
    "fp4_ragged": W.custom(4, 256, 512, [768, 0, 256, 1280], seed=115, fp4=True, b_major="k",
                           sf_format="ue8m0_32", input_order="ragged", out_dtype="bf16"),
    "fp4_ragged_split_k_f32": W.custom(2, 128, 256, [24576, 512], seed=116, fp4=True, b_major="k",
                                       sf_format="ue8m0_32", input_order="ragged"),
    # CTA-pair tiles (hidden 256) with the long expert split along K
    "fp4_pair_split_k_f32": W.custom(2, 256, 256, [32768, 512], seed=128, fp4=True, b_major="k",
                                     sf_format="ue8m0_32"),
    "nvfp4_pair_split_k_accumulate": W.custom(2, 256, 256, [32768, 512], seed=129, fp4=True, b_major="k",
                                              sf_format="ue4m3_16", accumulate=True),
    "fp8_general_scales_bf16": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=120, fp8=True, sf_format="f32_any",
                                        out_dtype="bf16"),
    "fp8_general_mn_a_k_b_accumulate_f32": W.custom(3, 256, 768, [256, 1280, 512], seed=121, fp8=True,
                                                    sf_format="f32_any", a_major="mn", b_major="k", accumulate=True),
    "fp8_general_ragged_discrete_f16": W.custom(3, 384, 512, [768, 256, 0], seed=122, fp8=True, sf_format="f32_any",
                                                input_order="ragged", output_mode="discrete", out_dtype="f16"),
    "fp8_general_long_expert_split_by_plan": W.custom(2, 128, 256, [32768, 256], seed=123, fp8=True,
                                                      sf_format="f32_any", accumulate=True, out_dtype="bf16"),
    "nvfp4_bf16_out": W.custom(4, 256, 512, [512, 0, 768, 1024], seed=117, fp4=True, b_major="k",
                               sf_format="ue4m3_16", out_dtype="bf16"),
    "nvfp4_split_k_f32_accumulate": W.custom(3, 128, 256, [32768, 0, 256], seed=118, fp4=True, b_major="k",
                                             sf_format="ue4m3_16", accumulate=True),
    "nvfp4_ragged_discrete_f16": W.custom(3, 256, 256, [1024, 512, 256], seed=119, fp4=True, b_major="k",
                                          sf_format="ue4m3_16", input_order="ragged", output_mode="discrete",
                                          out_dtype="f16"),
    "fp4_discrete_f16": W.custom(3, 256, 256, [1024, 512, 256], seed=113, fp4=True, b_major="k",
                                 sf_format="ue8m0_32", out_dtype="f16", output_mode="discrete"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_parity_small(name):
    _check(CASES[name])


def test_single_cta_and_pair_tiles_agree():
    """The same BF16 problem on 128-row single-CTA tiles and 256-row CTA-pair tiles."""
    kgw = ensure_built()
    w = W.custom(3, 512, 512, [1024, 256, 768], seed=67, out_dtype="bf16")
    x = W.make_inputs(w, DEV)
    pair = run_gpu(w, x, DEV).stacked().clone()
    prev = kgw.kgw_debug_set(3, 1)
    try:
        single = run_gpu(w, x, DEV).stacked().clone()
    finally:
        kgw.kgw_debug_set(3, prev)
    torch.cuda.synchronize()
    assert torch.equal(pair.view(torch.int16), single.view(torch.int16))


@pytest.mark.parametrize("fp8,hidden", [(False, 512), (False, 384), (True, 256)])
def test_storage_orders_are_bitwise_identical(fp8, hidden):
    """The same logical operands stored in all four orders give the same bits."""
    outs = []
    for am, bm in (("k", "mn"), ("mn", "mn"), ("k", "k"), ("mn", "k")):
        w = W.custom(3, hidden, 512, [768, 0, 1024], seed=96, fp8=fp8, a_major=am, b_major=bm, out_dtype="bf16")
        outs.append(run_gpu(w, W.make_inputs(w, DEV), DEV).stacked().clone())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))


def test_deterministic_bitwise():
    w = CASES["split_k_bf16_accumulate"]
    x = W.make_inputs(w, DEV)
    o1 = run_gpu(w, x, DEV).stacked().clone()
    o2 = run_gpu(w, x, DEV).stacked().clone()
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_dense_and_discrete_outputs_are_identical():
    w1 = W.custom(4, 256, 512, [512, 0, 256, 1024], seed=40, out_dtype="bf16")
    w2 = W.custom(4, 256, 512, [512, 0, 256, 1024], seed=40, out_dtype="bf16", output_mode="discrete")
    x = W.make_inputs(w1, DEV)
    a = run_gpu(w1, x, DEV).stacked()
    b = run_gpu(w2, x, DEV).stacked()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ragged_and_tensor2d_are_identical():
    counts = [768, 0, 1536, 256]
    w1 = W.custom(4, 256, 512, counts, seed=41)
    w2 = W.custom(4, 256, 512, counts, seed=41, input_order="ragged")
    x1 = W.make_inputs(w1, DEV)
    x2 = W.make_inputs(w2, DEV)
    assert torch.equal(x1.b, x2.b)
    a = run_gpu(w1, x1, DEV).stacked()
    b = run_gpu(w2, x2, DEV).stacked()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------------------------
# Device-detected errors: nothing is written
# ---------------------------------------------------------------------------------------------

def _bad_offsets_run(offsets_list, tokens_sum):
    kgw = ensure_built()
    w = W.custom(3, 128, 256, [256, 512, 768], seed=50)
    x = W.make_inputs(w, DEV)
    x.offsets = torch.tensor(offsets_list, dtype=torch.int32, device=DEV)
    outs = Outputs(w, DEV)
    before = outs.buf.clone()
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(3, 128, 256, tokens_sum, x.a, x.b, x.offsets, out=outs.dense, status_dev=status)
    ws = kgw.workspace_for(args, device=DEV)
    kgw.kgw_wgrad_bf16(args, ws)
    torch.cuda.synchronize()
    return int(status.item()), torch.equal(before, outs.buf)


@pytest.mark.parametrize("offsets", [[256, 128, 1536], [256, 700, 1536], [256, 768, 1280]])
def test_malformed_offsets_are_rejected_on_device(offsets):
    kgw = ensure_built()
    st, untouched = _bad_offsets_run(offsets, 1536)
    assert st == kgw.KGW_ERR_OFFSETS
    assert untouched


def test_bad_output_pointer_is_rejected_on_device():
    kgw = ensure_built()
    w = W.custom(3, 128, 256, [256, 512, 768], seed=51, output_mode="discrete")
    x = W.make_inputs(w, DEV)
    outs = Outputs(w, DEV)
    ptrs = outs.ptrs.clone()
    ptrs[1] = ptrs[1] + 8  # not 16-byte aligned
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    args = kgw.make_args(3, 128, 256, 1536, x.a, x.b, x.offsets, out_ptrs=ptrs, status_dev=status)
    kgw.kgw_wgrad_bf16(args, kgw.workspace_for(args, device=DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_ERR_OUT_PTRS
    assert all(torch.all(v == 7.25) for v in outs.views)


def test_host_rejects_unaligned_operand_on_gpu():
    kgw = ensure_built()
    w = W.tiny()
    x = W.make_inputs(w, DEV)
    outs = Outputs(w, DEV)
    ws = kgw.workspace_for(kgw.make_args(4, 128, 256, 1536, x.a, x.b, x.offsets, out=outs.dense), device=DEV)
    a_view = x.a.reshape(-1)[1:]  # 2-byte offset
    args = kgw.make_args(4, 128, 256, 1536, a_view, x.b, x.offsets, out=outs.dense)
    rc = kgw.kgw_wgrad_bf16(args, ws, check=False)
    assert rc == kgw.KGW_ERR_ALIGNMENT


def test_small_workspace_still_correct():
    """Down to the schedule alone (no room for split-K partials) the result is unchanged."""
    kgw = ensure_built()
    w = CASES["split_k"]
    x = W.make_inputs(w, DEV)
    full = run_gpu(w, x, DEV).stacked().clone()
    outs = Outputs(w, DEV)
    args = kgw.make_args(w.num_experts, w.hidden, w.intermediate, w.tokens_sum, x.a, x.b, x.offsets,
                         out=outs.dense)
    ws = torch.empty(64 * 1024, dtype=torch.uint8, device=DEV)
    kgw.kgw_wgrad_bf16(args, ws)
    torch.cuda.synchronize()
    x_cpu = W.make_inputs(w, "cpu")
    ref, S = oracle_full(w, x_cpu)
    assert_close_to_oracle(w, to_f64(outs.stacked()), ref, S)
    assert_close_to_oracle(w, to_f64(full), ref, S)
    assert not torch.equal(full, outs.stacked())  # split-K really changed the summation order


def test_fp4_rejects_unsupported_layouts():
    """FP4 needs K-major A and B (the packed-FP4 MMA reads K-major operands): an MN-major operand is
    KGW_ERR_UNSUPPORTED, host-side."""
    kgw = ensure_built()
    w = W.custom(2, 128, 256, [256, 256], seed=114, fp4=True, b_major="k", sf_format="ue8m0_32")
    x = W.make_inputs(w, DEV)
    out = torch.empty((2, 128, 256), dtype=torch.float32, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    for kw in ({"b_major": kgw.KGW_MN_MAJOR}, {"a_major": kgw.KGW_MN_MAJOR}):
        args = kgw.make_args(2, 128, 256, 512, x.a, x.b, x.offsets, out=out,
                             **{"b_major": kgw.KGW_K_MAJOR, **kw})
        assert kgw.kgw_wgrad_fp4_ue8m0(args, x.sfa, x.sfb, ws, check=False) == kgw.KGW_ERR_UNSUPPORTED


@pytest.mark.parametrize("hidden", [256, 384], ids=["pair", "single_cta"])
@pytest.mark.parametrize("kind", ["fp8_f32_nan", "fp8_ue8m0_nan", "fp4_ue8m0_nan", "nvfp4_sign_bit", "nvfp4_nan_byte"])
def test_bad_scales_are_reported(kind, hidden):
    """A NaN FP32 scale, a UE8M0 byte 0xFF (NaN) or an invalid UE4M3 byte (top bit set, or the NaN
    code 0x7F) anywhere in the scale tensors is reported as KGW_ERR_SCALES; clean scales report
    KGW_OK. Hidden 256 runs CTA pairs (the scale kernel checks the scales it prepares), hidden 384
    single CTAs (the converter warp checks them)."""
    kgw = ensure_built()
    H = hidden
    if kind == "fp8_f32_nan":
        w = W.custom(3, H, 512, [512, 256, 768], seed=140, fp8=True, out_dtype="bf16")
    elif kind == "fp8_ue8m0_nan":
        w = W.custom(3, H, 512, [512, 256, 768], seed=141, fp8=True, sf_format="ue8m0_32", out_dtype="bf16")
    elif kind == "fp4_ue8m0_nan":
        w = W.custom(3, H, 512, [512, 256, 768], seed=142, fp4=True, b_major="k", sf_format="ue8m0_32",
                     out_dtype="bf16")
    else:
        w = W.custom(3, H, 512, [512, 256, 768], seed=143, fp4=True, b_major="k", sf_format="ue4m3_16",
                     out_dtype="bf16")
    x = W.make_inputs(w, DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    run_gpu(w, x, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_OK
    # one bad entry, in B's scales of the last expert's last 128-token block, a column in the
    # second 128-column half of its n-tile, one byte that is not byte 0
    sfb = x.sfb.clone()
    if kind == "fp8_f32_nan":
        sfb[-1, 300] = float("nan")
    else:
        words = sfb.view(torch.int32)
        words[-1, 300] = int(np.array([0x7FFF7F7F], dtype=np.uint32).view(np.int32)[0])
    if kind == "nvfp4_sign_bit":
        words[-1, 300] = int(np.array([0x38B83838], dtype=np.uint32).view(np.int32)[0])   # 0xB8: sign bit set
    if kind == "nvfp4_nan_byte":
        words[-1, 300] = int(np.array([0x387F3838], dtype=np.uint32).view(np.int32)[0])   # 0x7F: UE4M3 NaN
    x2 = W.Inputs(x.a, x.b, x.offsets, x.sfa, sfb, x.c, x.gsa, x.gsb)
    status.fill_(-1)
    run_gpu(w, x2, DEV, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_ERR_SCALES


def test_fp8_scales_that_are_not_powers_of_two_take_the_promotion_path():
    """The same e4m3 operands with one scale changed from a power of two to 3x it: no error, the
    result follows the oracle, and it is exactly 3x the original for the block that scale covers."""
    kgw = ensure_built()
    w = W.custom(2, 128, 256, [256, 256], seed=124, fp8=True)
    x = W.make_inputs(w, DEV)
    x_cpu = W.make_inputs(w, "cpu")
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    base = run_gpu(w, x, DEV, status=status).stacked().clone()
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_OK
    sfa = x.sfa.clone()
    sfa[:, 5] *= 3.0                       # every block of A's row 5: not a power of two any more
    x2 = W.Inputs(x.a, x.b, x.offsets, sfa, x.sfb, x.c)
    status.fill_(-1)
    got = run_gpu(w, x2, DEV, status=status).stacked().clone()
    torch.cuda.synchronize()
    assert int(status.item()) == kgw.KGW_OK
    x2c = W.Inputs(x_cpu.a, x_cpu.b, x_cpu.offsets, sfa.cpu(), x_cpu.sfb, x_cpu.c)
    ref, S = oracle_full(w, x2c)
    assert_close_to_oracle(w, to_f64(got), ref, S)
    others = torch.ones(128, dtype=torch.bool)
    others[5] = False
    # (different kernels sum in different orders: equal up to FP32 accumulation, not bit for bit)
    assert torch.allclose(got[:, 5, :], 3.0 * base[:, 5, :], rtol=1e-5, atol=1e-3)
    assert torch.allclose(got[:, others, :], base[:, others, :], rtol=1e-5, atol=1e-3)


@pytest.mark.parametrize("kw", [dict(), dict(sf_format="ue8m0_32", a_major="mn", b_major="k"),
                                dict(input_order="ragged", out_dtype="bf16"), dict(sf_format="f32_any")],
                         ids=["f32_scales", "ue8m0_mn_a_k_b", "ragged_bf16", "general_scales"])
def test_fp8_pair_tiles_agree_with_single_cta_tiles(kw):
    """FP8 problems whose hidden size is a multiple of 256 run on CTA pairs (256 x 256 tiles, scale
    factors prepared by the scale kernel); the same call forced onto single-CTA 128 x 256 tiles
    gives the same result within the FP32 accumulation bound, and both match the oracle."""
    kgw = ensure_built()
    w = W.custom(3, 512, 512, [768, 0, 1280], seed=125, fp8=True, **kw)
    x = W.make_inputs(w, DEV)
    x_cpu = W.make_inputs(w, "cpu")
    pair = run_gpu(w, x, DEV).stacked().clone()
    prev = kgw.kgw_debug_set(3, 1)
    try:
        single = run_gpu(w, x, DEV).stacked().clone()
    finally:
        kgw.kgw_debug_set(3, prev)
    torch.cuda.synchronize()
    ref, S = oracle_full(w, x_cpu)
    assert_close_to_oracle(w, to_f64(pair), ref, S)
    assert_close_to_oracle(w, to_f64(single), ref, S)


@pytest.mark.parametrize("kw", [dict(out_dtype="bf16"), dict(input_order="ragged", accumulate=True),
                                dict(unaligned=True, out_dtype="bf16"),
                                dict(sf_format="ue4m3_16", out_dtype="bf16"),
                                dict(sf_format="ue4m3_16", input_order="ragged")],
                         ids=["tensor2d_bf16", "ragged_accumulate_f32", "unaligned_counts", "nvfp4_tensor2d_bf16",
                              "nvfp4_ragged_f32"])
def test_fp4_pair_tiles_agree_with_single_cta_tiles(kw):
    """FP4 and NVFP4 problems whose hidden size is a multiple of 256 run on CTA pairs (scale
    factors prepared by the scale kernel: two 128-token blocks per stage, NVFP4 four 64-token
    words); forced onto single-CTA tiles they give the same result within the FP32 accumulation
    bound, and both match the oracle. The unaligned case ends experts on a stage that holds a
    single scale block (384 and 96 tokens)."""
    kgw = ensure_built()
    counts = [384, 0, 1280, 96] if kw.get("unaligned") else [768, 0, 1280, 512]
    kw = dict(kw)
    sf_format = kw.pop("sf_format", "ue8m0_32")
    w = W.custom(4, 512, 512, counts, seed=127, fp4=True, b_major="k", sf_format=sf_format, **kw)
    x = W.make_inputs(w, DEV)
    x_cpu = W.make_inputs(w, "cpu")
    pair = run_gpu(w, x, DEV).stacked().clone()
    prev = kgw.kgw_debug_set(3, 1)
    try:
        single = run_gpu(w, x, DEV).stacked().clone()
    finally:
        kgw.kgw_debug_set(3, prev)
    torch.cuda.synchronize()
    ref, S = oracle_full(w, x_cpu)
    assert_close_to_oracle(w, to_f64(pair), ref, S)
    assert_close_to_oracle(w, to_f64(single), ref, S)
