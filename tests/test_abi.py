"""The C ABI: the library builds, loads, exports every declared symbol, and the host-side
argument checks reject bad calls before touching the GPU (no compute call here)."""
import ctypes

import pytest
import torch

from kgw_testlib import HEADER, ensure_built, header_functions

kgw = ensure_built()


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("kgw_workspace_size", "kgw_wgrad_bf16", "kgw_wgrad_fp8_blockscaled", "kgw_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = kgw.lib()
    for name in header_functions():
        assert hasattr(L, name), name


def test_binding_has_the_same_names():
    for name in header_functions():
        assert callable(getattr(kgw, name)), name


def test_status_strings():
    assert kgw.kgw_status_string(0) == "KGW_OK"
    assert kgw.kgw_status_string(6) == "KGW_ERR_OFFSETS"
    assert kgw.kgw_status_string(999) == "KGW_ERR_UNKNOWN"
    assert kgw.kgw_version() >= 100


def test_struct_layout_matches_header():
    # int32 x3, int64, ptr, int32, ptr, int32, ptr, int32, ptr, ptr, int32, int32, ptr
    assert ctypes.sizeof(kgw.KgwArgs) == 104


FAKE = 1 << 20  # 16-byte aligned fake device address (never dereferenced by the host checks)


def good_args(**kw):
    base = dict(num_experts=4, hidden=128, intermediate=256, tokens_sum=1536, a=FAKE, b=FAKE, offsets=FAKE,
                out=FAKE)
    base.update(kw)
    return kgw.make_args(base.pop("num_experts"), base.pop("hidden"), base.pop("intermediate"),
                         base.pop("tokens_sum"), base.pop("a"), base.pop("b"), base.pop("offsets"), **base)


def rc_bf16(args, ws=FAKE, nbytes=1 << 30):
    return kgw.lib().kgw_wgrad_bf16(ctypes.byref(args), ws, nbytes, None)


def test_workspace_size_is_host_only_and_monotone():
    small = kgw.kgw_workspace_size(good_args())
    big = kgw.kgw_workspace_size(good_args(hidden=4096, intermediate=2048, tokens_sum=33792, num_experts=8))
    assert 0 < small < big
    assert big <= 256 * 2 * 128 * 256 * 4 + (1 << 20)  # at most 256 partial tiles of 256 x 256 FP32


@pytest.mark.parametrize("kw,code", [
    (dict(num_experts=0), kgw.KGW_ERR_INVALID_ARG),
    (dict(num_experts=5000), kgw.KGW_ERR_INVALID_ARG),
    (dict(hidden=100), kgw.KGW_ERR_UNSUPPORTED),
    (dict(intermediate=128), kgw.KGW_ERR_UNSUPPORTED),
    (dict(tokens_sum=1000), kgw.KGW_ERR_INVALID_ARG),
    (dict(tokens_sum=-256), kgw.KGW_ERR_INVALID_ARG),
    (dict(a_major=7), kgw.KGW_ERR_INVALID_ARG),
    (dict(input_order=5), kgw.KGW_ERR_INVALID_ARG),
    (dict(out_dtype=3), kgw.KGW_ERR_INVALID_ARG),
    (dict(offsets=None), kgw.KGW_ERR_INVALID_ARG),
    (dict(out=None), kgw.KGW_ERR_INVALID_ARG),                  # neither output
    (dict(out_ptrs=FAKE), kgw.KGW_ERR_INVALID_ARG),             # both outputs
    (dict(out=FAKE + 8), kgw.KGW_ERR_ALIGNMENT),
    (dict(a=FAKE + 2), kgw.KGW_ERR_ALIGNMENT),
    (dict(b=FAKE + 4), kgw.KGW_ERR_ALIGNMENT),
    (dict(a=None), kgw.KGW_ERR_INVALID_ARG),
])
def test_host_validation(kw, code):
    args = good_args(**kw)
    assert rc_bf16(args) == code
    # the sizing call takes any token total (it also sizes kgw_wgrad_bf16_unaligned calls)
    if (code != kgw.KGW_ERR_UNSUPPORTED or "hidden" in kw or "intermediate" in kw) and kw.get("tokens_sum") != 1000:
        n = ctypes.c_size_t(0)
        assert kgw.lib().kgw_workspace_size(ctypes.byref(args), 0, ctypes.byref(n)) == code


@pytest.mark.parametrize("a_major,b_major,tokens_sum,code", [
    (0, 1, 1000, None),                       # K-major A: multiples of 8 pass host validation
    (0, 1, 1001, kgw.KGW_ERR_INVALID_ARG),
    (1, 0, 1004, kgw.KGW_ERR_INVALID_ARG),    # K-major B: likewise
    (1, 1, 1001, None),                       # both MN-major: any count
])
def test_unaligned_entry_token_rule(a_major, b_major, tokens_sum, code):
    """kgw_wgrad_bf16_unaligned: host-side token-total rule (no device work is enqueued on CPU;
    a passing call gets as far as the device check, which fails here without a GPU)."""
    args = good_args(a_major=a_major, b_major=b_major, tokens_sum=tokens_sum)
    rc = kgw.lib().kgw_wgrad_bf16_unaligned(ctypes.byref(args), FAKE, 1 << 30, None)
    if code is None:
        assert rc in (kgw.KGW_ERR_DEVICE, kgw.KGW_ERR_CUDA)
    else:
        assert rc == code
    n = ctypes.c_size_t(0)
    assert kgw.lib().kgw_workspace_size(ctypes.byref(args), 0, ctypes.byref(n)) == kgw.KGW_OK


@pytest.mark.parametrize("a_major,b_major", [(0, 1), (1, 1), (0, 0), (1, 0)])
def test_all_four_operand_orders_pass_host_validation(a_major, b_major):
    args = good_args(a_major=a_major, b_major=b_major)
    assert kgw.kgw_workspace_size(args) > 0


def test_workspace_checks():
    args = good_args()
    assert rc_bf16(args, ws=None) == kgw.KGW_ERR_WORKSPACE
    assert rc_bf16(args, ws=FAKE + 16) == kgw.KGW_ERR_WORKSPACE
    assert rc_bf16(args, nbytes=64) == kgw.KGW_ERR_WORKSPACE


def test_null_args_pointer():
    assert kgw.lib().kgw_wgrad_bf16(None, FAKE, 1 << 20, None) == kgw.KGW_ERR_INVALID_ARG


def test_fp8_entry_needs_scales():
    args = good_args()
    rc = kgw.lib().kgw_wgrad_fp8_blockscaled(ctypes.byref(args), None, None, FAKE, 1 << 30, None)
    assert rc in (kgw.KGW_ERR_INVALID_ARG, kgw.KGW_ERR_UNSUPPORTED)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_device_reports_device_error():
    assert rc_bf16(good_args()) == kgw.KGW_ERR_DEVICE


def test_debug_hooks_roundtrip():
    prev = kgw.kgw_debug_set(1, 123456789)
    assert kgw.kgw_debug_set(1, prev) == 123456789
    assert kgw.kgw_debug_set(99, 0) == -1


def test_binding_constants_match_the_header():
    """Every enumerator of include/kgw.h has the same value in the Python binding."""
    import re
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    found = re.findall(r"\b(KGW_[A-Z0-9_]+)\s*=\s*(\d+)", src)
    assert len(found) >= 15
    for name, value in found:
        assert getattr(kgw, name) == int(value), name


def test_noalloc_rejects_more_experts_than_its_scratch_holds():
    """The entry point without a workspace keeps its scratch in a fixed static array: more than
    1024 experts is rejected on the host, before any device query or launch."""
    args = good_args(num_experts=1025, tokens_sum=256)
    assert kgw.lib().kgw_wgrad_bf16_noalloc(ctypes.byref(args), None) == kgw.KGW_ERR_SCRATCH_LIMIT
    bad = good_args(num_experts=1024, hidden=100)
    assert kgw.lib().kgw_wgrad_bf16_noalloc(ctypes.byref(bad), None) == kgw.KGW_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["fp8", "fp4", "nvfp4"])
def test_block_scaled_pairs_need_room_for_the_prepared_scale_factors(entry):
    """Block-scaled calls on CTA pairs (hidden % 256 == 0) keep their scale factors, prepared in
    TMEM order, in the workspace: a workspace that holds only the schedule is KGW_ERR_WORKSPACE on
    the host, before any device query, while a BF16 call of the same shape passes with it; the size
    kgw_workspace_size gives (is_fp8 = 1) passes the host checks, and the call then stops at the
    device check here, without a GPU."""
    args = good_args(hidden=256, tokens_sum=65536, b_major=kgw.KGW_K_MAJOR)
    L = kgw.lib()
    small = 64 * 1024   # the schedule of 4 experts fits; 516 prepared scale rows of 512 words do not

    def call(nbytes):
        if entry == "fp8":
            return L.kgw_wgrad_fp8_blockscaled(ctypes.byref(args), FAKE, FAKE, FAKE, nbytes, None)
        if entry == "fp4":
            return L.kgw_wgrad_fp4_ue8m0(ctypes.byref(args), FAKE, FAKE, FAKE, nbytes, None)
        return L.kgw_wgrad_nvfp4(ctypes.byref(args), FAKE, FAKE, None, None, FAKE, nbytes, None)

    assert call(small) == kgw.KGW_ERR_WORKSPACE
    assert rc_bf16(args, nbytes=small) in (kgw.KGW_ERR_DEVICE, kgw.KGW_ERR_CUDA)
    assert call(kgw.kgw_workspace_size(args, True)) in (kgw.KGW_ERR_DEVICE, kgw.KGW_ERR_CUDA)
