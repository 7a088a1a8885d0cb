"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The CUDA path computes every output; the oracle recomputes every output too, one expert at a
time from the stored operands (``expert_from_storage``: that expert's A and B decoded to
float64, scaled per token block for FP8/FP4, multiplied in float64), so memory stays bounded by
one expert. Every element is compared with the per-element bound; empty experts are checked
exactly: zeros when overwriting, the pre-filled output bit for bit when accumulating. Each test
prints the worst err/tol it saw.
"""
import dataclasses

import pytest

import workloads as W
from kgw_testlib import check_full

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_full_balanced_bf16():
    check_full(W.balanced(), "balanced")


def test_full_wide_accumulate_bf16():
    check_full(W.wide(), "wide")


def test_full_skewed_ragged_discrete():
    check_full(W.skewed(), "skewed")


def test_full_fp8_blockscaled():
    check_full(W.fp8(), "fp8")


def test_full_fp8_ue8m0_gran32():
    check_full(dataclasses.replace(W.fp8(), sf_format="ue8m0_32"), "fp8 ue8m0 gran 32")


def test_full_balanced_token_major_a():
    """The balanced workload with A = dY^T read from dY stored token-major (M-major A)."""
    check_full(dataclasses.replace(W.balanced(), a_major="mn"), "balanced, M-major A")


def test_full_fp4_blockscaled():
    """FP4 e2m1 operands with UE8M0 scales per 32 tokens, at the FP8 workload's shape."""
    check_full(W.fp4(), "fp4")


def test_full_nvfp4():
    """NVFP4 (UE4M3 scales per 16 tokens, FP32 global scales) at the FP8 workload's shape."""
    check_full(W.nvfp4(), "nvfp4")


def test_full_fp8_general_fp32_scales():
    """FP8 with FP32 scales amax/448 (not powers of two): the promotion path at full size."""
    check_full(W.fp8_fp32(), "fp8 general FP32 scales")
