"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to something the pages or mathematics fix: exact rational
brute force, the block-masked dense GEMM identity, closed forms, special cases that
reduce to a plain library GEMM, the empty-expert and accumulate semantics of
"Grouped GEMM + WGrad (Unified)" (section "Operation"), the offsets contract (section
"BF16 contract"), and the exact decoding of the stored number formats.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.kgw_oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def e4m3_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def random_bf16(rng, shape, choices=None):
    if choices is None:
        x = rng.standard_normal(shape).astype(np.float32)
    else:
        x = rng.choice(np.asarray(choices, dtype=np.float32), size=shape)
    return torch.from_numpy(x).to(torch.bfloat16)


# ------------------------------------------------------------------------------------------
# Number formats
# ------------------------------------------------------------------------------------------

def test_bf16_decode_known_values():
    known = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0000: 0.0, 0x3F00: 0.5,
             0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127}
    bits = np.array(list(known.keys()), dtype=np.uint16)
    got = O.bf16_to_f64(bits)
    assert got.tolist() == list(known.values())


def test_bf16_decode_all_patterns_vs_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # the signalling-NaN patterns are decoded too
        got = O.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_known_values():
    known = {0x38: 1.0, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6,
             0x07: 7 * 2.0 ** -9, 0x40: 2.0, 0x3C: 1.5, 0x00: 0.0}
    got = O.e4m3_to_f64(np.array(list(known.keys()), dtype=np.uint8))
    assert got.tolist() == list(known.values())
    assert np.isnan(O.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------------------------------------
# Offsets contract
# ------------------------------------------------------------------------------------------

def _read_golden_offsets():
    rows = []
    with open(os.path.join(GOLDEN, "contract_offsets.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            ts, offs, valid, why = [p.strip() for p in line.split("|")]
            rows.append((int(ts), [int(v) for v in offs.split()], bool(int(valid)), why))
    return rows


@pytest.mark.parametrize("case", _read_golden_offsets(), ids=lambda c: c[3])
def test_offsets_contract_golden(case):
    tokens_sum, offsets, valid, _ = case
    assert O.offsets_valid(np.array(offsets, dtype=np.int32), tokens_sum) == valid


def test_howto_example_counts_rejected():
    kv = {}
    with open(os.path.join(GOLDEN, "howto_example_counts.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            kv[k] = [int(x) for x in v]
    counts = np.array(kv["tokens_per_expert"])
    assert len(counts) == kv["num_experts"][0]
    offsets = np.cumsum(counts)
    assert O.offsets_valid(offsets, int(counts.sum())) == bool(kv["valid"][0])


def test_expert_ranges_definition():
    assert O.expert_ranges([256, 768, 768, 1536]) == [(0, 256), (256, 768), (768, 768), (768, 1536)]


# ------------------------------------------------------------------------------------------
# Exact brute force (Fraction) on tiny shapes
# ------------------------------------------------------------------------------------------

def _fraction_wgrad(A, B, offsets, C=None):
    """Exact rational per-expert product, written as a plain triple loop."""
    H, T = A.shape
    I = B.shape[1]
    fa = [[Fraction(float(A[m, k])) for k in range(T)] for m in range(H)]
    fb = [[Fraction(float(B[k, n])) for n in range(I)] for k in range(T)]
    out = []
    prev = 0
    for e, end in enumerate([int(v) for v in offsets]):
        res = [[Fraction(0) if C is None else Fraction(float(C[e][m][n])) for n in range(I)]
               for m in range(H)]
        for m in range(H):
            for n in range(I):
                s = res[m][n]
                for k in range(prev, end):
                    s += fa[m][k] * fb[k][n]
                res[m][n] = s
        out.append(res)
        prev = end
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_exact_fraction_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    E, H, I = 3, 5, 4
    counts = np.array([256, 0, 512])[rng.permutation(3)]
    offsets = np.cumsum(counts)
    T = int(offsets[-1])
    a = random_bf16(rng, (H, T))
    b = random_bf16(rng, (T, I))
    out, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    A = a.to(torch.float64).numpy()
    B = b.to(torch.float64).numpy()
    exact = _fraction_wgrad(A, B, offsets)
    for e in range(E):
        for m in range(H):
            for n in range(I):
                err = abs(Fraction(out[e, m, n]) - exact[e][m][n])
                assert err <= Fraction(1e-12) * Fraction(S[e, m, n]) + Fraction(1e-300)


def test_oracle_accumulate_matches_exact_fraction():
    rng = np.random.default_rng(7)
    E, H, I = 2, 3, 3
    offsets = np.array([256, 256])
    a = random_bf16(rng, (H, 256))
    b = random_bf16(rng, (256, I))
    C = rng.standard_normal((E, H, I))
    out, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I, c_init=C, accumulate=True)
    exact = _fraction_wgrad(a.to(torch.float64).numpy(), b.to(torch.float64).numpy(), offsets, C)
    for e in range(E):
        for m in range(H):
            for n in range(I):
                err = abs(Fraction(out[e, m, n]) - exact[e][m][n])
                assert err <= Fraction(1e-12) * (Fraction(S[e, m, n]) + abs(Fraction(C[e, m, n]))) + Fraction(1e-300)
    # empty expert (index 1) keeps C bit for bit
    assert np.array_equal(out[1], C[1])


# ------------------------------------------------------------------------------------------
# Identities that tie the per-expert product to a plain dense GEMM (torch float64 matmul)
# ------------------------------------------------------------------------------------------

def _case(seed, counts, H=24, I=40):
    rng = np.random.default_rng(seed)
    offsets = np.cumsum(counts).astype(np.int32)
    T = int(offsets[-1])
    a = random_bf16(rng, (H, T))
    b = random_bf16(rng, (T, I))
    return a, b, offsets


def test_block_masked_dense_identity():
    counts = [512, 256, 0, 768, 256]
    a, b, offsets = _case(11, counts)
    H, I = a.shape[0], b.shape[1]
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    A = a.to(torch.float64)
    B = b.to(torch.float64)
    begin = 0
    total = torch.zeros(H, I, dtype=torch.float64)
    for e, n in enumerate(counts):
        mask = torch.zeros(A.shape[1], dtype=torch.float64)
        mask[begin:begin + n] = 1.0
        masked = (A * mask) @ B                     # dense GEMM over the whole token axis
        S = A.abs() @ B.abs()
        assert torch.all((torch.from_numpy(out[e]) - masked).abs() <= 1e-12 * S + 1e-300)
        total += torch.from_numpy(out[e])
        begin += n
    dense = A @ B
    assert torch.allclose(total, dense, rtol=0, atol=1e-10 * float((A.abs() @ B.abs()).max()))


def test_single_expert_is_plain_gemm():
    a, b, offsets = _case(12, [1024])
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, a.shape[0], b.shape[1])
    ref = (a.to(torch.float64) @ b.to(torch.float64)).numpy()
    assert np.allclose(out[0], ref, rtol=0, atol=1e-12 * np.abs(ref).max() * 100)


def test_empty_expert_overwrite_gives_zeros_and_accumulate_keeps_c():
    a, b, offsets = _case(13, [256, 0, 512, 0])
    H, I = a.shape[0], b.shape[1]
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    assert not out[1].any() and not out[3].any()
    C = np.random.default_rng(1).standard_normal((4, H, I))
    acc, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I, c_init=C, accumulate=True)
    assert np.array_equal(acc[1], C[1]) and np.array_equal(acc[3], C[3])


def test_accumulate_equals_c_plus_overwrite():
    a, b, offsets = _case(14, [256, 768])
    H, I = a.shape[0], b.shape[1]
    # integer-valued C so that C + R is exact in float64 for this small K
    C = np.random.default_rng(2).integers(-4, 5, size=(2, H, I)).astype(np.float64)
    ow, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    acc, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I, c_init=C, accumulate=True)
    assert np.allclose(acc, C + ow, rtol=0, atol=1e-9)


def test_splitting_an_expert_sums_to_merged():
    a, b, offsets_split = _case(15, [256, 512, 256])
    H, I = a.shape[0], b.shape[1]
    merged = np.array([256, 1024], dtype=np.int32)            # experts 1+2 merged
    r_split, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets_split, H, I)
    r_merged, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), merged, H, I)
    assert np.array_equal(r_split[0], r_merged[0])
    assert np.all(np.abs(r_split[1] + r_split[2] - r_merged[1]) <= 1e-12 * (S[1] + S[2]) + 1e-300)


def test_token_permutation_within_expert_is_invariant():
    counts = [512, 768]
    a, b, offsets = _case(16, counts)
    H, I = a.shape[0], b.shape[1]
    perm = np.concatenate([np.random.default_rng(3).permutation(512),
                           512 + np.random.default_rng(4).permutation(768)])
    a2 = a[:, perm].contiguous()
    b2 = b[perm, :].contiguous()
    r1, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    r2, _ = O.wgrad_from_storage(bf16_bits(a2), bf16_bits(b2), offsets, H, I)
    assert np.all(np.abs(r1 - r2) <= 1e-12 * S + 1e-300)


def test_permuting_tokens_across_experts_changes_result():
    """Sanity for the pins above: moving tokens between experts must change the result."""
    a, b, offsets = _case(17, [256, 256])
    H, I = a.shape[0], b.shape[1]
    perm = np.concatenate([np.arange(256, 512), np.arange(0, 256)])
    r1, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    r2, _ = O.wgrad_from_storage(bf16_bits(a[:, perm].contiguous()), bf16_bits(b[perm].contiguous()),
                                 offsets, H, I)
    assert not np.allclose(r1, r2)
    assert np.allclose(r1[0], r2[1]) and np.allclose(r1[1], r2[0])


def test_ragged_equals_tensor2d_on_same_logical_values():
    counts = [256, 0, 768, 512]
    a, b, offsets = _case(18, counts)
    H, I = a.shape[0], b.shape[1]
    ragged = W.pack_ragged_a(a, np.array(counts))
    r2d, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I, input_order="tensor2d")
    rrg, _ = O.wgrad_from_storage(bf16_bits(ragged), bf16_bits(b), offsets, H, I, input_order="ragged")
    assert np.array_equal(r2d, rrg)
    # and the ragged storage really is different memory order (leading dimension n_e)
    assert not np.array_equal(bf16_bits(ragged), bf16_bits(a).reshape(-1))


# ------------------------------------------------------------------------------------------
# Closed forms
# ------------------------------------------------------------------------------------------

def test_ones_closed_form():
    counts = [256, 0, 512, 1024]
    offsets = np.cumsum(counts)
    H, I = 8, 16
    T = int(offsets[-1])
    a = torch.ones(H, T, dtype=torch.bfloat16)
    b = torch.ones(T, I, dtype=torch.bfloat16)
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    for e, n in enumerate(counts):
        assert np.all(out[e] == float(n))


def test_rank_one_closed_form_detects_transposition():
    """A[m,k] = a_m and B[k,n] = b_n give R_e[m,n] = n_e * a_m * b_n exactly."""
    counts = [256, 512, 0]
    offsets = np.cumsum(counts)
    H, I = 6, 10
    T = int(offsets[-1])
    am = np.array([1, -2, 0.5, 3, -0.25, 1.5], dtype=np.float32)
    bn = np.linspace(-2, 2, I).astype(np.float32)
    a = torch.from_numpy(np.repeat(am[:, None], T, axis=1)).to(torch.bfloat16)
    b = torch.from_numpy(np.repeat(bn[None, :], T, axis=0)).to(torch.bfloat16)
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    av = a[:, 0].to(torch.float64).numpy()
    bv = b[0, :].to(torch.float64).numpy()
    for e, n in enumerate(counts):
        assert np.array_equal(out[e], n * np.outer(av, bv))


def test_one_hot_selects_rows_of_b():
    """A[m,k] = [k == begin_e + m] picks row begin_e + m of B for expert e."""
    counts = [256, 512]
    offsets = np.cumsum(counts)
    H, I = 4, 12
    T = int(offsets[-1])
    rng = np.random.default_rng(5)
    b = random_bf16(rng, (T, I))
    a = torch.zeros(H, T, dtype=torch.bfloat16)
    begins = [0, 256]
    for bgn in begins:
        for m in range(H):
            a[m, bgn + 3 * m + 1] = 1.0
    out, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    B = b.to(torch.float64).numpy()
    for e, bgn in enumerate(begins):
        for m in range(H):
            assert np.array_equal(out[e, m], B[bgn + 3 * m + 1])


# ------------------------------------------------------------------------------------------
# FP8 block-scaled variant
# ------------------------------------------------------------------------------------------

def _fp8_case(seed, counts, H=16, I=24):
    offsets = np.cumsum(counts).astype(np.int32)
    T = int(offsets[-1])
    g = torch.Generator().manual_seed(seed)
    a32 = torch.randn(H, T, generator=g)
    b32 = torch.randn(T, I, generator=g)
    qa, sfa = W.quantize_e4m3_blocks(a32, token_axis=1)
    qb, sfb = W.quantize_e4m3_blocks(b32, token_axis=0)
    return qa, sfa, qb, sfb, offsets


def test_fp8_unit_scales_equal_decoded_product():
    qa, sfa, qb, sfb, offsets = _fp8_case(21, [256, 0, 512])
    H, I = qa.shape[0], qb.shape[1]
    ones_a = torch.ones_like(sfa)
    ones_b = torch.ones_like(sfb)
    r, _ = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), offsets, H, I, fp8=True,
                                sfa=ones_a.numpy(), sfb=ones_b.numpy())
    A = qa.to(torch.float64)
    B = qb.to(torch.float64)
    begin = 0
    for e, end in enumerate(offsets.tolist()):
        ref = (A[:, begin:end] @ B[begin:end]).numpy()
        assert np.allclose(r[e], ref, rtol=0, atol=1e-9)
        begin = end


def test_fp8_block_scale_power_of_two_is_exact():
    """Scaling one 128-token block's A scales by 2**j scales that block's contribution by 2**j."""
    qa, sfa, qb, sfb, offsets = _fp8_case(22, [256])
    H, I = qa.shape[0], qb.shape[1]
    # zero every token outside block 1 so that the result is that block's contribution alone
    qa_only = qa.clone()
    qa_only[:, :128] = 0
    base, _ = O.wgrad_from_storage(e4m3_bits(qa_only), e4m3_bits(qb), offsets, H, I, fp8=True,
                                   sfa=sfa.numpy(), sfb=sfb.numpy())
    sfa2 = sfa.clone()
    sfa2[1, :] *= 2.0 ** 5
    scaled, _ = O.wgrad_from_storage(e4m3_bits(qa_only), e4m3_bits(qb), offsets, H, I, fp8=True,
                                     sfa=sfa2.numpy(), sfb=sfb.numpy())
    assert np.array_equal(scaled, base * 2.0 ** 5)


def test_fp8_scale_indexing_row_vs_column():
    """A's scale is per (block, row m); B's is per (block, column n): a closed form."""
    H, I, T = 3, 5, 256
    offsets = np.array([T], dtype=np.int32)
    qa = torch.ones(H, T).to(torch.float8_e4m3fn)
    qb = torch.ones(T, I).to(torch.float8_e4m3fn)
    sfa = np.array([[1.0, 2.0, 4.0], [8.0, 16.0, 32.0]], dtype=np.float32)        # [2, H]
    sfb = np.array([[1.0, 0.5, 0.25, 2.0, 4.0], [1.0, 1.0, 1.0, 1.0, 1.0]], dtype=np.float32)  # [2, I]
    r, _ = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), offsets, H, I, fp8=True, sfa=sfa, sfb=sfb)
    expect = 128 * (np.outer(sfa[0], sfb[0]) + np.outer(sfa[1], sfb[1]))
    assert np.array_equal(r[0], expect)


def test_fp8_quantiser_is_in_range_and_power_of_two():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(8, 512, generator=g) * 3
    q, s = W.quantize_e4m3_blocks(x, token_axis=1)
    s = s.numpy()
    mant, _ = np.frexp(s)
    assert np.all(mant == 0.5)                                    # powers of two
    dec = O.e4m3_to_f64(e4m3_bits(q))
    assert np.all(np.abs(dec) <= 448)
    recon = O.apply_scales_rows(dec, s, 128)
    # e4m3 keeps 3 mantissa bits: relative error <= 2**-4 (plus subnormal floor)
    err = np.abs(recon - x.numpy().astype(np.float64))
    assert np.all(err <= 2.0 ** -4 * np.abs(x.numpy()) + np.repeat(s.T, 128, axis=1) * 2.0 ** -10)


# ------------------------------------------------------------------------------------------
# Tolerance
# ------------------------------------------------------------------------------------------

def test_bf16_rounding_of_reference_is_within_tolerance():
    a, b, offsets = _case(31, [256, 512])
    H, I = a.shape[0], b.shape[1]
    ref, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    rounded = torch.from_numpy(ref).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(rounded - ref) <= O.tolerance(S, ref, "bf16"))
    # and the bound is not vacuous: a 1% error is rejected somewhere
    assert np.any(np.abs(ref * 1.01 - ref) > O.tolerance(S, ref, "f32"))


# ------------------------------------------------------------------------------------------
# Planted mistakes: each pin above must catch a plausible bug planted in the oracle
# ------------------------------------------------------------------------------------------

def _brute_force_agrees(fn_ranges=None, transpose_b=False):
    rng = np.random.default_rng(99)
    H, I = 4, 4
    offsets = np.array([256, 512])
    a = random_bf16(rng, (H, 512))
    b = random_bf16(rng, (512, I))
    bb = bf16_bits(b)
    if transpose_b:
        bb = bb.reshape(512, I)[:, ::-1].copy()
    out, S = O.wgrad_from_storage(bf16_bits(a), bb, offsets, H, I)
    exact = _fraction_wgrad(a.to(torch.float64).numpy(), b.to(torch.float64).numpy(), offsets)
    for e in range(2):
        for m in range(H):
            for n in range(I):
                if abs(Fraction(out[e, m, n]) - exact[e][m][n]) > Fraction(1e-12) * Fraction(S[e, m, n]) + Fraction(1e-300):
                    return False
    return True


def test_planted_range_bug_is_caught(monkeypatch):
    assert _brute_force_agrees()
    good = O.expert_ranges

    def off_by_one(offsets):
        return [(b + (1 if e > 0 else 0), end) for e, (b, end) in enumerate(good(offsets))]

    monkeypatch.setattr(O, "expert_ranges", off_by_one)
    assert not _brute_force_agrees()


def test_planted_operand_bug_is_caught():
    assert not _brute_force_agrees(transpose_b=True)


def test_planted_ragged_bug_is_caught(monkeypatch):
    counts = [256, 512]
    a, b, offsets = _case(41, counts, H=8, I=8)
    ragged = W.pack_ragged_a(a, np.array(counts))
    good = O.logical_a

    def wrong_ld(a_values, hidden, offsets_, order, a_major="k"):
        if order != "ragged":
            return good(a_values, hidden, offsets_, order, a_major)
        # bug: treat the ragged buffer as if it had leading dimension tokens_sum
        return np.asarray(a_values).reshape(hidden, -1)

    r_ok, _ = O.wgrad_from_storage(bf16_bits(ragged), bf16_bits(b), offsets, 8, 8, input_order="ragged")
    O.logical_a = wrong_ld
    try:
        r_bad, _ = O.wgrad_from_storage(bf16_bits(ragged), bf16_bits(b), offsets, 8, 8, input_order="ragged")
    finally:
        O.logical_a = good
    r_2d, _ = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, 8, 8)
    assert np.array_equal(r_ok, r_2d)
    assert not np.array_equal(r_bad, r_2d)


@pytest.mark.parametrize("order", ["tensor2d", "ragged"])
def test_element_from_storage_matches_full_oracle(order):
    counts = [256, 0, 512, 768]
    a, b, offsets = _case(51, counts, H=8, I=12)
    H, I = 8, 12
    a_store = a if order == "tensor2d" else W.pack_ragged_a(a, np.array(counts))
    full, S = O.wgrad_from_storage(bf16_bits(a_store), bf16_bits(b), offsets, H, I, input_order=order)
    for (e, m, n) in [(0, 0, 0), (2, 7, 11), (3, 3, 5), (1, 2, 2), (3, 7, 0)]:
        v, s = O.element_from_storage(bf16_bits(a_store), bf16_bits(b), offsets, H, I, e, m, n, input_order=order)
        assert abs(v - full[e, m, n]) <= 1e-12 * S[e, m, n] + 1e-300
        assert abs(s - S[e, m, n]) <= 1e-12 * S[e, m, n] + 1e-300


def test_element_from_storage_fp8():
    qa, sfa, qb, sfb, offsets = _fp8_case(52, [256, 0, 512])
    H, I = qa.shape[0], qb.shape[1]
    full, S = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), offsets, H, I, fp8=True,
                                   sfa=sfa.numpy(), sfb=sfb.numpy())
    for (e, m, n) in [(0, 1, 2), (2, 15, 23), (1, 0, 0)]:
        v, s = O.element_from_storage(e4m3_bits(qa), e4m3_bits(qb), offsets, H, I, e, m, n, fp8=True,
                                      sfa=sfa.numpy(), sfb=sfb.numpy())
        assert abs(v - full[e, m, n]) <= 1e-12 * S[e, m, n] + 1e-300


# ------------------------------------------------------------------------------------------
# Operand storage orders ("Grouped GEMM + WGrad (Unified)", section "BF16 contract": A K-major or
# M-major, B K-major or N-major; ragged keeps each operand's unit-stride axis)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("order", ["tensor2d", "ragged"])
@pytest.mark.parametrize("a_major,b_major", [("k", "mn"), ("mn", "mn"), ("k", "k"), ("mn", "k")])
def test_storage_orders_give_the_same_result(order, a_major, b_major):
    counts = [256, 0, 768, 512]
    w = W.custom(4, 16, 24, counts, seed=61, input_order=order, a_major=a_major, b_major=b_major)
    ref_w = W.custom(4, 16, 24, counts, seed=61)
    x = W.make_inputs(w)
    x0 = W.make_inputs(ref_w)
    r, S = O.wgrad_from_storage(bf16_bits(x.a), bf16_bits(x.b), x.offsets.numpy(), 16, 24, input_order=order,
                                a_major=a_major, b_major=b_major)
    r0, _ = O.wgrad_from_storage(bf16_bits(x0.a), bf16_bits(x0.b), x0.offsets.numpy(), 16, 24)
    assert np.array_equal(r, r0)
    # the stored bytes really differ from the K-major/N-major tensor2d layout unless nothing moved
    if (a_major, b_major, order) != ("k", "mn", "tensor2d"):
        same_a = bf16_bits(x.a).size == bf16_bits(x0.a).size and np.array_equal(bf16_bits(x.a).ravel(), bf16_bits(x0.a).ravel())
        same_b = np.array_equal(bf16_bits(x.b).ravel(), bf16_bits(x0.b).ravel())
        assert not (same_a and same_b)
    for (e, m, n) in [(0, 3, 5), (2, 15, 23), (3, 0, 0)]:
        v, s = O.element_from_storage(bf16_bits(x.a), bf16_bits(x.b), x.offsets.numpy(), 16, 24, e, m, n,
                                      input_order=order, a_major=a_major, b_major=b_major)
        assert abs(v - r[e, m, n]) <= 1e-12 * S[e, m, n] + 1e-300


def test_mn_major_a_is_the_transpose_in_memory():
    """M-major A stores A^T contiguously: element (m, k) at k*hidden + m."""
    H, T = 8, 256
    a = torch.arange(H * T, dtype=torch.float32).reshape(H, T).to(torch.bfloat16)
    w = W.custom(1, H, 16, [T], seed=0, a_major="mn")
    a_store, _ = W.store_operands(w, a, torch.zeros(T, 16, dtype=torch.bfloat16))
    flat = a_store.reshape(-1)
    for (m, k) in [(0, 0), (3, 17), (7, 255)]:
        assert flat[k * H + m] == a[m, k]
    L = O.logical_a(bf16_bits(a_store), H, np.array([T]), "tensor2d", "mn")
    assert np.array_equal(L, bf16_bits(a).reshape(H, T))


def test_f16_rounding_of_reference_is_within_tolerance():
    a, b, offsets = _case(32, [256, 512])
    H, I = a.shape[0], b.shape[1]
    ref, S = O.wgrad_from_storage(bf16_bits(a), bf16_bits(b), offsets, H, I)
    rounded = torch.from_numpy(ref).to(torch.float32).to(torch.float16).to(torch.float64).numpy()
    assert np.all(np.abs(rounded - ref) <= O.tolerance(S, ref, "f16"))
    # FP16 keeps 3 more mantissa bits than BF16: its bound is tighter
    assert np.all(O.tolerance(S, ref, "f16") <= O.tolerance(S, ref, "bf16") + 2.0 ** -24)



# ------------------------------------------------------------------------------------------
# Packed UE8M0 scales, 32-token granularity
# ------------------------------------------------------------------------------------------

def test_ue8m0_unpack_known_words():
    w = np.array([[127 | (128 << 8) | (126 << 16) | (0 << 24)]], dtype=np.uint32).view(np.int32)
    s = O.unpack_ue8m0_32(w)
    assert s[:, 0].tolist() == [1.0, 2.0, 0.5, 2.0 ** -127]


def test_ue8m0_each_32_token_block_has_its_own_scale():
    """Ones x ones with block scales 2^(j) on A's 32-token block j: R = 32 * sum_j 2^j * sb_j."""
    H, I, T = 2, 3, 128
    qa = torch.ones(H, T).to(torch.float8_e4m3fn)
    qb = torch.ones(T, I).to(torch.float8_e4m3fn)
    wa = np.array([[127 | (128 << 8) | (129 << 16) | (130 << 24)] * H], dtype=np.uint32).view(np.int32)
    wb = np.array([[127 | (127 << 8) | (127 << 16) | (131 << 24)] * I], dtype=np.uint32).view(np.int32)
    r, _ = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), np.array([T]), H, I, fp8=True, sfa=wa, sfb=wb,
                                sf_format="ue8m0_32")
    expect = 32 * (1 * 1 + 2 * 1 + 4 * 1 + 8 * 16)
    assert np.all(r[0] == expect)


def test_ue8m0_equal_subblocks_match_fp32_per_128_scales():
    g = torch.Generator().manual_seed(5)
    H, I, T = 8, 16, 256
    qa = (torch.randn(H, T, generator=g) * 4).to(torch.float8_e4m3fn)
    qb = (torch.randn(T, I, generator=g) * 4).to(torch.float8_e4m3fn)
    ka = np.random.default_rng(1).integers(-5, 6, size=(2, H))
    kb = np.random.default_rng(2).integers(-5, 6, size=(2, I))
    def pack(k):
        b = (k + 127).astype(np.uint32)
        return (b | (b << 8) | (b << 16) | (b << 24)).view(np.int32)
    r32, _ = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), np.array([T]), H, I, fp8=True,
                                  sfa=pack(ka), sfb=pack(kb), sf_format="ue8m0_32")
    r128, _ = O.wgrad_from_storage(e4m3_bits(qa), e4m3_bits(qb), np.array([T]), H, I, fp8=True,
                                   sfa=np.ldexp(1.0, ka).astype(np.float32), sfb=np.ldexp(1.0, kb).astype(np.float32))
    assert np.array_equal(r32, r128)


def test_ue8m0_quantiser_recipe():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4, 256, generator=g) * 3
    q, packed = W.quantize_e4m3_ue8m0_32(x, token_axis=1)
    s = O.unpack_ue8m0_32(packed.numpy())           # [8, 4]
    dec = O.e4m3_to_f64(e4m3_bits(q))
    assert np.all(np.abs(dec) <= 448)
    recon = O.apply_scales_rows(dec, s, 32)
    err = np.abs(recon - x.numpy().astype(np.float64))
    assert np.all(err <= 2.0 ** -4 * np.abs(x.numpy()) + np.repeat(s.T, 32, axis=1) * 2.0 ** -10)


# ------------------------------------------------------------------------------------------
# FP4 (e2m1 elements, UE8M0 scales per 32 tokens)
# ------------------------------------------------------------------------------------------

def _fp4_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_codes.txt")) if l.strip() and not l.startswith("#")]
    return {int(c, 16): float(v) for c, v in rows}


def test_e2m1_decode_matches_format_table():
    table = _fp4_golden()
    codes = np.arange(16, dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)   # low nibble = first element
    got = O.e2m1_to_f64(packed)
    for c in range(16):
        assert got[c] == table[c] and np.signbit(got[c]) == np.signbit(table[c]), c


def test_e2m1_nibble_order():
    assert O.e2m1_to_f64(np.array([0x21], dtype=np.uint8)).tolist() == [0.5, 1.0]
    assert O.e2m1_to_f64(np.array([0x7F], dtype=np.uint8)).tolist() == [-6.0, 6.0]


def test_fp4_quantiser_round_trip_on_grid():
    """Values that are grid points times a power of two come back exactly, with their scale."""
    rng = np.random.default_rng(31)
    grid = np.array(sorted(set(_fp4_golden().values())))
    k = rng.integers(-6, 6, size=(3, 8))                       # one exponent per 32-token block
    vals = rng.choice(grid, size=(3, 256))
    vals[:, ::32] = 6.0                                        # amax of every block is 6 * 2**k
    x = vals * np.ldexp(1.0, np.repeat(k, 32, axis=1))
    q, sf = W.quantize_e2m1_ue8m0_32(torch.from_numpy(x.astype(np.float32)), token_axis=1)
    dec = O.e2m1_to_f64(q.numpy()).reshape(3, 256)
    scales = O.unpack_ue8m0_32(sf.numpy())                     # [256/32, 3]
    assert np.array_equal(dec * np.repeat(scales.T, 32, axis=1), x)


def test_fp4_unit_scales_equal_bf16_oracle():
    """FP4 with all scales 1 is the BF16 operation on the decoded values (all e2m1 values are
    exact in bf16): ties the FP4 decoding and layout to the independently pinned BF16 path."""
    rng = np.random.default_rng(32)
    counts = [256, 0, 512]
    offs = np.cumsum(counts).astype(np.int32)
    T, H, I = 768, 8, 16
    codes_a = rng.integers(0, 16, size=(H, T)).astype(np.uint8)
    codes_b = rng.integers(0, 16, size=(I, T)).astype(np.uint8)         # K-major B [I, T]
    pa = codes_a[:, 0::2] | (codes_a[:, 1::2] << 4)
    pb = codes_b[:, 0::2] | (codes_b[:, 1::2] << 4)
    ones_a = np.full((T // 128, H), 0x7F7F7F7F, dtype=np.uint32).view(np.int32)
    ones_b = np.full((T // 128, I), 0x7F7F7F7F, dtype=np.uint32).view(np.int32)
    got, S = O.wgrad_from_storage(pa, pb, offs, H, I, fp4=True, sfa=ones_a, sfb=ones_b, b_major="k",
                                  sf_format="ue8m0_32")
    table = _fp4_golden()
    va = np.vectorize(table.get)(codes_a).astype(np.float32)
    vb = np.vectorize(table.get)(codes_b).astype(np.float32)
    a16 = torch.from_numpy(va).to(torch.bfloat16)
    b16 = torch.from_numpy(vb.T.copy()).to(torch.bfloat16)                # N-major [T, I]
    ref, S2 = O.wgrad_from_storage(bf16_bits(a16), bf16_bits(b16), offs, H, I)
    assert np.array_equal(got, ref) and np.array_equal(S, S2)


def test_fp4_brute_force_with_scales():
    rng = np.random.default_rng(33)
    counts = [256, 256]
    offs = np.cumsum(counts).astype(np.int32)
    T, H, I = 512, 2, 3
    codes_a = rng.integers(0, 16, size=(H, T)).astype(np.uint8)
    codes_b = rng.integers(0, 16, size=(I, T)).astype(np.uint8)
    pa = codes_a[:, 0::2] | (codes_a[:, 1::2] << 4)
    pb = codes_b[:, 0::2] | (codes_b[:, 1::2] << 4)
    ea = rng.integers(120, 135, size=(T // 32, H))
    eb = rng.integers(120, 135, size=(T // 32, I))

    def pack(e):
        e = e.astype(np.uint32).reshape(T // 128, 4, -1)
        return (e[:, 0] | (e[:, 1] << 8) | (e[:, 2] << 16) | (e[:, 3] << 24)).view(np.int32)

    got, _ = O.wgrad_from_storage(pa, pb, offs, H, I, fp4=True, sfa=pack(ea), sfb=pack(eb), b_major="k",
                                  sf_format="ue8m0_32")
    table = {c: Fraction(v) for c, v in _fp4_golden().items()}
    for e, (b, end) in enumerate([(0, 256), (256, 512)]):
        for m in range(H):
            for n in range(I):
                exact = sum(table[int(codes_a[m, k])] * Fraction(2) ** int(ea[k // 32, m] - 127) *
                            table[int(codes_b[n, k])] * Fraction(2) ** int(eb[k // 32, n] - 127)
                            for k in range(b, end))
                assert Fraction(got[e, m, n]) == exact


def test_fp4_element_from_storage_matches_full():
    w = W.custom(3, 128, 256, [256, 0, 512], seed=34, fp4=True, b_major="k", sf_format="ue8m0_32",
                 out_dtype="bf16")
    x = W.make_inputs(w, "cpu")
    full, S = O.wgrad_from_storage(x.a.numpy(), x.b.numpy(), w.offsets, 128, 256, fp4=True, sfa=x.sfa.numpy(),
                                   sfb=x.sfb.numpy(), b_major="k", sf_format="ue8m0_32")
    for (e, m, n) in [(0, 0, 0), (0, 127, 255), (2, 64, 17), (2, 3, 200)]:
        v, s = O.element_from_storage(x.a.numpy(), x.b.numpy(), w.offsets, 128, 256, e, m, n, fp4=True,
                                      sfa=x.sfa.numpy(), sfb=x.sfb.numpy(), b_major="k", sf_format="ue8m0_32")
        assert abs(v - full[e, m, n]) <= 1e-12 * (1 + S[e, m, n]) and abs(s - S[e, m, n]) <= 1e-12 * (1 + S[e, m, n])


# ------------------------------------------------------------------------------------------
# One expert at a time (the full-size parity tests compare every element this way)
# ------------------------------------------------------------------------------------------

_EXPERT_CASES = [
    dict(),
    dict(input_order="ragged"),
    dict(a_major="mn"),
    dict(b_major="k"),
    dict(input_order="ragged", a_major="mn", b_major="k"),
    dict(input_order="ragged", b_major="k"),
    dict(fp8=True),
    dict(fp8=True, sf_format="ue8m0_32", input_order="ragged"),
    dict(fp8=True, a_major="mn", b_major="k"),
    dict(fp4=True, b_major="k", sf_format="ue8m0_32"),
    dict(fp4=True, b_major="k", sf_format="ue8m0_32", input_order="ragged"),
]


def test_fp4_ragged_order_is_the_same_problem_as_tensor2d():
    """Ragged FP4 stores each expert's [rows, n_e/2]-byte block back to back; the oracle reads the same
    logical values as from the tensor2d layout, and the stored bytes really moved."""
    kw = dict(fp4=True, b_major="k", sf_format="ue8m0_32")
    counts = [256, 0, 512, 768]
    w2 = W.custom(4, 128, 256, counts, seed=83, **kw)
    wr = W.custom(4, 128, 256, counts, seed=83, input_order="ragged", **kw)
    x2, xr = W.make_inputs(w2, "cpu"), W.make_inputs(wr, "cpu")
    assert not np.array_equal(x2.a.numpy().ravel(), xr.a.numpy().ravel())
    common = dict(fp4=True, b_major="k", sf_format="ue8m0_32", sfa=x2.sfa.numpy(), sfb=x2.sfb.numpy())
    r2, _ = O.wgrad_from_storage(x2.a.numpy(), x2.b.numpy(), w2.offsets, 128, 256, **common)
    rr, _ = O.wgrad_from_storage(xr.a.numpy(), xr.b.numpy(), wr.offsets, 128, 256, input_order="ragged", **common)
    assert np.array_equal(r2, rr)


@pytest.mark.parametrize("kw", _EXPERT_CASES, ids=lambda kw: "-".join(f"{k}={v}" for k, v in kw.items()) or "bf16")
def test_expert_from_storage_matches_whole_problem(kw):
    """Each expert's (R_e, S_e) read straight from storage equals the whole-problem oracle's."""
    counts = [256, 0, 512, 768]
    w = W.custom(4, 128, 256, counts, seed=81, **kw)
    x = W.make_inputs(w, "cpu")
    if w.fp8 or w.fp4:
        bits = lambda t: t.contiguous().view(torch.uint8).numpy()
    else:
        bits = bf16_bits
    sf = dict(sfa=None if x.sfa is None else x.sfa.numpy(), sfb=None if x.sfb is None else x.sfb.numpy())
    common = dict(input_order=w.input_order, fp8=w.fp8, a_major=w.a_major, b_major=w.b_major,
                  sf_format=w.sf_format, fp4=w.fp4, **sf)
    full, S = O.wgrad_from_storage(bits(x.a), bits(x.b), w.offsets, 128, 256, **common)
    for e in range(4):
        r, s = O.expert_from_storage(bits(x.a), bits(x.b), w.offsets, 128, 256, e, **common)
        assert r.shape == (128, 256) and s.shape == (128, 256)
        assert np.all(np.abs(r - full[e]) <= 1e-12 * S[e] + 1e-300)
        assert np.all(np.abs(s - S[e]) <= 1e-12 * S[e] + 1e-300)
    assert not np.any(O.expert_from_storage(bits(x.a), bits(x.b), w.offsets, 128, 256, 1, **common)[0])


def test_expert_from_storage_catches_a_shifted_expert():
    """Reading expert e's neighbour (an off-by-one expert index in the addressing) must differ."""
    counts = [256, 512, 768]
    w = W.custom(3, 128, 256, counts, seed=82, input_order="ragged")
    x = W.make_inputs(w, "cpu")
    full, S = O.wgrad_from_storage(bf16_bits(x.a), bf16_bits(x.b), w.offsets, 128, 256, input_order="ragged")
    r, _ = O.expert_from_storage(bf16_bits(x.a), bf16_bits(x.b), w.offsets, 128, 256, 1, input_order="ragged")
    assert np.all(np.abs(r - full[1]) <= 1e-12 * S[1] + 1e-300)
    assert not np.allclose(r, full[2][:, :]) and not np.allclose(r, full[0])


# ------------------------------------------------------------------------------------------
# Scale blocks per expert (counts that are not multiples of 128): each expert's 128-token blocks
# start at its first token ("05 · Grouped GEMM 与 Expert 计算", section 4: every expert segment is
# padded to the quantisation alignment before the FP8/FP4 cast)
# ------------------------------------------------------------------------------------------

def test_token_scale_rows_by_hand():
    rows = O.token_scale_rows([40, 40, 240], 128)            # counts 40, 0, 200
    assert rows.tolist() == [0] * 40 + [1] * 128 + [2] * 72
    rows32 = O.token_scale_rows([40, 40, 240], 32)
    assert rows32.tolist() == [0] * 32 + [1] * 8 + sum(([4 + j] * 32 for j in range(6)), []) + [10] * 8
    # multiples of 128: the global blocks k // block
    offs = np.cumsum([256, 0, 384, 128])
    for blk in (32, 128):
        assert np.array_equal(O.token_scale_rows(offs, blk), np.arange(768) // blk)


def _fp8_brute(codes_a, codes_b, sa, sb, counts):
    """Exact sum over each expert's tokens of dec(a)*sa[block]*dec(b)*sb[block], with blocks counted
    from each expert's first token (written out with explicit loops, independently of the oracle)."""
    table = {c: Fraction(float(v)) for c, v in enumerate(O.e4m3_to_f64(np.arange(256, dtype=np.uint8)))
             if np.isfinite(v)}
    H, I = codes_a.shape[0], codes_b.shape[1]
    out, b, sblk = [], 0, 0
    for n in counts:
        res = [[Fraction(0)] * I for _ in range(H)]
        for j in range(n):
            k, blk = b + j, sblk + j // 128
            for m in range(H):
                fa = table[int(codes_a[m, k])] * Fraction(float(sa[blk, m]))
                for c in range(I):
                    res[m][c] += fa * table[int(codes_b[k, c])] * Fraction(float(sb[blk, c]))
        out.append(res)
        b += n
        sblk += -(-n // 128)
    return out


def test_fp8_per_expert_blocks_brute_force():
    rng = np.random.default_rng(41)
    counts = [48, 0, 176, 16]                                  # multiples of 16, not of 128
    T, H, I = sum(counts), 3, 4
    nblk = sum(-(-n // 128) for n in counts)                   # 1 + 0 + 2 + 1
    codes_a = rng.integers(0, 126, size=(H, T)).astype(np.uint8)   # finite codes only
    codes_b = rng.integers(0, 126, size=(T, I)).astype(np.uint8)
    sa = np.ldexp(1.0, rng.integers(-6, 7, size=(nblk, H))).astype(np.float32)
    sb = np.ldexp(1.0, rng.integers(-6, 7, size=(nblk, I))).astype(np.float32)
    offs = np.cumsum(counts).astype(np.int32)
    got, S = O.wgrad_from_storage(codes_a, codes_b, offs, H, I, fp8=True, sfa=sa, sfb=sb)
    exact = _fp8_brute(codes_a, codes_b, sa, sb, counts)
    for e in range(len(counts)):
        for m in range(H):
            for n in range(I):
                assert abs(Fraction(got[e, m, n]) - exact[e][m][n]) <= Fraction(1e-12) * Fraction(S[e, m, n]) + Fraction(1e-300)
    # the same numbers through the one-expert and one-element readers
    for e in range(len(counts)):
        r, _ = O.expert_from_storage(codes_a, codes_b, offs, H, I, e, fp8=True, sfa=sa, sfb=sb)
        assert np.all(np.abs(r - got[e]) <= 1e-12 * S[e] + 1e-300)
        v, _ = O.element_from_storage(codes_a, codes_b, offs, H, I, e, H - 1, I - 1, fp8=True, sfa=sa, sfb=sb)
        assert abs(v - got[e, H - 1, I - 1]) <= 1e-12 * S[e, H - 1, I - 1] + 1e-300


@pytest.mark.parametrize("kind", ["fp8", "fp8_ue8m0", "fp4"])
def test_per_expert_quantisation_roundtrip_needs_per_expert_scale_rows(kind):
    """Decoding the quantised operands with the oracle's per-expert scale rows gives back the
    drawn values within the element format's precision; reading the scales at global rows
    k // 128 instead (a plausible indexing mistake) does not."""
    counts = [48, 0, 176, 96] if kind != "fp4" else [64, 0, 160, 96]
    kw = dict(fp8=True) if kind == "fp8" else (dict(fp8=True, sf_format="ue8m0_32") if kind == "fp8_ue8m0" else
                                                dict(fp4=True, b_major="k", sf_format="ue8m0_32"))
    w = W.custom(4, 128, 256, counts, seed=42, unaligned=True, **kw)
    x = W.make_inputs(w, "cpu")
    g = torch.Generator().manual_seed(42)
    a32 = torch.randn(128, w.tokens_sum, generator=g).double().numpy()
    dec = O.e2m1_to_f64 if w.fp4 else O.e4m3_to_f64
    bits = x.a.contiguous().view(torch.uint8).numpy()
    a = dec(bits).reshape(128, w.tokens_sum)
    sa, blk = O.decode_scales(x.sfa.numpy(), w.sf_format)
    good = O.apply_scales_rows(a, sa, blk, O.token_scale_rows(w.offsets, blk))
    # half a unit in the last place of the element format, relative, plus half its smallest step
    # (e2m1: 0.5; e4m3: 2**-9) times the element's scale for values that round towards zero
    rel, step = (2.0 ** -2, 0.5) if w.fp4 else (2.0 ** -4, 2.0 ** -9)
    rows = O.token_scale_rows(w.offsets, blk)
    floor = 0.5 * step * O.apply_scales_rows(np.ones_like(a), sa, blk, rows)
    assert np.all(np.abs(good - a32) <= rel * np.abs(a32) + floor)
    rows_global = np.minimum(np.arange(w.tokens_sum) // blk, sa.shape[0] - 1)
    bad = O.apply_scales_rows(a, sa, blk, rows_global)
    assert not np.all(np.abs(bad - a32) <= rel * np.abs(a32) + floor)


# ------------------------------------------------------------------------------------------
# NVFP4: e2m1 elements, unsigned-E4M3 scales per 16 tokens, FP32 global scales (the cuDNN page's
# block-scaled contract: sf_vec_size 16 and global_scale_a / global_scale_b)
# ------------------------------------------------------------------------------------------

def test_ue4m3_decoder_matches_torch_e4m3_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = O.ue4m3_to_f64(codes)
    ref = torch.from_numpy(codes[:128].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got[:127], ref[:127])                 # 0x00..0x7E: the e4m3 values
    assert np.isnan(got[127]) and np.all(np.isnan(got[128:]))   # 0x7F NaN; a sign bit is invalid
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[1] == 2.0 ** -9


def test_ue4m3_words_unpack_to_16_token_rows():
    w = np.array([[0x38403038, 0x7E000001]], dtype=np.uint32).view(np.int32)     # [1 word-row, 2 columns]
    s = O.unpack_ue4m3_16(w)
    assert s.shape == (4, 2)
    assert s[:, 0].tolist() == [1.0, 0.5, 2.0, 1.0]       # bytes 0x38, 0x30, 0x40, 0x38
    assert s[:, 1].tolist() == [2.0 ** -9, 0.0, 0.0, 448.0]


def test_nvfp4_quantiser_round_trip():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(64, 512, generator=g) * 5
    gs = W.nvfp4_global_scale(x)
    q, words = W.quantize_e2m1_ue4m3_16(x, 1, gs)
    s, blk = O.decode_scales(words.numpy(), "ue4m3_16")
    assert blk == 16 and not np.isnan(s).any() and s.max() <= 448
    dec = O.apply_scales_rows(O.e2m1_to_f64(q.numpy()).reshape(64, 512), s, 16) * gs
    per = O.apply_scales_rows(np.ones((64, 512)), s, 16) * gs
    err = np.abs(dec - x.double().numpy())
    assert np.all(err <= 2.0 ** -2 * np.abs(x.double().numpy()) + 0.25 * per + 1e-12)
    # scales are the smallest E4M3 values that cover each block's amax / 6
    amax = np.abs(x.double().numpy()).reshape(64, 32, 16).max(axis=2).T           # [blocks, rows]
    assert np.all(s * gs * 6 >= amax * (1 - 2.0 ** -23))


def test_nvfp4_brute_force_with_global_scales():
    rng = np.random.default_rng(44)
    counts = [128, 0, 128]
    T, H, I = 256, 2, 3
    offs = np.cumsum(counts).astype(np.int32)
    codes_a = rng.integers(0, 16, size=(H, T)).astype(np.uint8)
    codes_b = rng.integers(0, 16, size=(I, T)).astype(np.uint8)
    pa = codes_a[:, 0::2] | (codes_a[:, 1::2] << 4)
    pb = codes_b[:, 0::2] | (codes_b[:, 1::2] << 4)
    sa_codes = rng.integers(0x20, 0x50, size=(T // 16, H)).astype(np.uint32)
    sb_codes = rng.integers(0x20, 0x50, size=(T // 16, I)).astype(np.uint32)

    def pack(c):
        c = c.reshape(T // 64, 4, -1)
        return (c[:, 0] | (c[:, 1] << 8) | (c[:, 2] << 16) | (c[:, 3] << 24)).view(np.int32)

    ga, gb = np.float32(0.375), np.float32(-1.25)
    got, S = O.wgrad_from_storage(pa, pb, offs, H, I, fp4=True, b_major="k", sf_format="ue4m3_16",
                                  sfa=pack(sa_codes), sfb=pack(sb_codes), global_scale_a=ga, global_scale_b=gb)
    e2m1 = {c: Fraction(v) for c, v in _fp4_golden().items()}
    e4m3 = lambda c: Fraction(float(torch.tensor([int(c)], dtype=torch.uint8).view(torch.float8_e4m3fn).double()))
    g = Fraction(float(ga)) * Fraction(float(gb))
    for e, (b, end) in enumerate([(0, 128), (128, 128), (128, 256)]):
        for m in range(H):
            for n in range(I):
                exact = g * sum(e2m1[int(codes_a[m, k])] * e4m3(sa_codes[k // 16, m]) *
                                e2m1[int(codes_b[n, k])] * e4m3(sb_codes[k // 16, n]) for k in range(b, end))
                assert abs(Fraction(got[e, m, n]) - exact) <= Fraction(1e-12) * Fraction(S[e, m, n]) + Fraction(1e-300)
    # the global scales multiply exactly: doubling one doubles every result
    got2, _ = O.wgrad_from_storage(pa, pb, offs, H, I, fp4=True, b_major="k", sf_format="ue4m3_16",
                                   sfa=pack(sa_codes), sfb=pack(sb_codes), global_scale_a=2 * ga, global_scale_b=gb)
    assert np.array_equal(got2, 2 * got)


# ------------------------------------------------------------------------------------------
# General FP32 scales ("05 · Grouped GEMM 与 Expert 计算", section 3: x_scales float)
# ------------------------------------------------------------------------------------------

def test_general_fp32_scale_quantiser_round_trip():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(16, 512, generator=g) * 7
    q, s = W.quantize_e4m3_fp32_blocks(x, token_axis=1)
    s = s.numpy()
    mant, _ = np.frexp(s)
    assert np.mean(mant != 0.5) > 0.9                       # not powers of two
    dec = O.e4m3_to_f64(e4m3_bits(q))
    assert np.all(np.abs(dec) <= 448) and np.all(np.isfinite(dec))
    recon = O.apply_scales_rows(dec, s, 128)
    err = np.abs(recon - x.numpy().astype(np.float64))
    assert np.all(err <= 2.0 ** -4 * np.abs(x.numpy()) + np.repeat(s.T, 128, axis=1) * 2.0 ** -10)


def test_fp8_brute_force_with_general_fp32_scales():
    rng = np.random.default_rng(45)
    counts = [128, 256]
    T, H, I = 384, 2, 3
    codes_a = rng.integers(0, 126, size=(H, T)).astype(np.uint8)
    codes_b = rng.integers(0, 126, size=(T, I)).astype(np.uint8)
    sa = rng.uniform(0.01, 3.0, size=(T // 128, H)).astype(np.float32)
    sb = (rng.uniform(-2.0, 2.0, size=(T // 128, I))).astype(np.float32)   # negative and fractional scales
    offs = np.cumsum(counts).astype(np.int32)
    got, S = O.wgrad_from_storage(codes_a, codes_b, offs, H, I, fp8=True, sfa=sa, sfb=sb, sf_format="f32_any")
    exact = _fp8_brute(codes_a, codes_b, sa, sb, counts)
    for e in range(2):
        for m in range(H):
            for n in range(I):
                assert abs(Fraction(got[e, m, n]) - exact[e][m][n]) <= Fraction(1e-12) * Fraction(S[e, m, n]) + Fraction(1e-300)
