"""The M-grouped entry points' host-side checks (no GPU needed): argument rules, workspace sizing,
and that a well-formed call gets as far as the device check. Nothing here dereferences the fake
device addresses: every case is decided before the library touches the GPU."""
import ctypes

import pytest
import torch

from kgw_testlib import ensure_built

kgw = ensure_built()
FAKE = 1 << 20          # 256-byte aligned fake device address
L = kgw.lib()


def mg_args(G=2, m=256, n=256, k=128, **kw):
    base = dict(a=FAKE, b=FAKE, groups=FAKE, d=FAKE)
    base.update(kw)
    return kgw.make_mgrouped_args(G, m, n, k, base.pop("a"), base.pop("b"), base.pop("groups"), base.pop("d"),
                                  **base)


def rc_bf16(args, ws=FAKE, nbytes=1 << 30):
    return L.kgw_mgrouped_bf16(ctypes.byref(args), ws, nbytes, None)


def rc_fp8(args, sfa=FAKE, sfb=FAKE, fmt=0, ws=FAKE, nbytes=1 << 30):
    return L.kgw_mgrouped_fp8(ctypes.byref(args), sfa, sfb, fmt, ws, nbytes, None)


def ws_size(args):
    n = ctypes.c_size_t(0)
    rc = L.kgw_mgrouped_workspace_size(ctypes.byref(args), ctypes.byref(n))
    return rc, n.value


def test_struct_layout_matches_header():
    # int32 num_groups, layout, m, n, k; ptr a, b; int32 b_major; ptr groups, d; int32 out_dtype,
    # accumulate; ptr status_dev
    assert ctypes.sizeof(kgw.KgwMgroupedArgs) == 80


@pytest.mark.parametrize("kw,code", [
    (dict(n=128), kgw.KGW_ERR_UNSUPPORTED),                  # n % 256
    (dict(k=96), kgw.KGW_ERR_UNSUPPORTED),                   # k % 64
    (dict(m=200), kgw.KGW_ERR_INVALID_ARG),                  # contiguous rows in whole 128-row tiles
    (dict(G=0), kgw.KGW_ERR_INVALID_ARG),
    (dict(G=5000), kgw.KGW_ERR_INVALID_ARG),                 # at most 4096 groups
    (dict(m=-128), kgw.KGW_ERR_INVALID_ARG),
    (dict(layout=7), kgw.KGW_ERR_INVALID_ARG),
    (dict(out_dtype=9), kgw.KGW_ERR_INVALID_ARG),
    (dict(b_major=4), kgw.KGW_ERR_INVALID_ARG),
    (dict(groups=None), kgw.KGW_ERR_INVALID_ARG),            # no group description
    (dict(b=None), kgw.KGW_ERR_INVALID_ARG),
    (dict(a=None), kgw.KGW_ERR_INVALID_ARG),
    (dict(d=None), kgw.KGW_ERR_INVALID_ARG),
    (dict(a=FAKE + 2), kgw.KGW_ERR_ALIGNMENT),
    (dict(b=FAKE + 8), kgw.KGW_ERR_ALIGNMENT),
    (dict(d=FAKE + 4), kgw.KGW_ERR_ALIGNMENT),
    (dict(groups=FAKE + 2), kgw.KGW_ERR_ALIGNMENT),
])
def test_host_rules(kw, code):
    args = mg_args(**kw)
    assert rc_bf16(args) == code
    assert ws_size(args)[0] == code


def test_masked_rows_need_no_alignment_and_size_by_groups():
    ok = mg_args(G=3, m=200, layout=kgw.KGW_MG_MASKED)      # max_m needs no alignment when masked
    assert ws_size(ok)[0] == kgw.KGW_OK
    rc1, small = ws_size(mg_args(G=2, m=256))
    rc2, big = ws_size(mg_args(G=2, m=256 * 64))
    assert rc1 == rc2 == kgw.KGW_OK and 0 < small < big


def test_index_layout_without_rows_needs_no_ids():
    # m = 0 rows: nothing to compute, so no per-row ids, A or D are needed
    args = mg_args(m=0, layout=kgw.KGW_MG_INDICES, groups=None, a=None, d=None)
    assert ws_size(args)[0] == kgw.KGW_OK


def test_workspace_rules():
    args = mg_args()
    assert rc_bf16(args, ws=0) == kgw.KGW_ERR_WORKSPACE
    assert rc_bf16(args, ws=FAKE + 16) == kgw.KGW_ERR_WORKSPACE
    assert rc_bf16(args, nbytes=16) == kgw.KGW_ERR_WORKSPACE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_well_formed_calls_stop_at_the_device_check():
    assert rc_bf16(mg_args()) == kgw.KGW_ERR_DEVICE
    assert rc_fp8(mg_args(k=128)) == kgw.KGW_ERR_DEVICE


def test_fp8_host_rules():
    assert rc_fp8(mg_args(k=192)) == kgw.KGW_ERR_UNSUPPORTED          # k % 128
    assert rc_fp8(mg_args(k=128), sfa=0) == kgw.KGW_ERR_INVALID_ARG     # scales required
    assert rc_fp8(mg_args(k=128), sfb=0) == kgw.KGW_ERR_INVALID_ARG
    assert rc_fp8(mg_args(k=128), sfa=FAKE + 4) == kgw.KGW_ERR_ALIGNMENT
    assert rc_fp8(mg_args(k=128), fmt=5) == kgw.KGW_ERR_INVALID_ARG     # FP32 (0) or packed UE8M0 (1)
