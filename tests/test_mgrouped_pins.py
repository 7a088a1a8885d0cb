"""Pins for the M-grouped GEMM oracle: checks against things other than the oracle itself.

Exact rational brute force; special cases that reduce to a plain library GEMM; closed forms;
equivalences between the three row layouts of "05 · Grouped GEMM 与 Expert 计算" section 2
(contiguous with offsets, contiguous with per-row group ids, masked); the masked semantics
(only the first masked_m rows are written, section 2.2); and the forward / dgrad / wgrad
identities of section 5 that tie the M-grouped oracle to the independently pinned K-grouped one.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.kgw_oracle as KO
import oracle.mgrouped_oracle as MO
import workloads.mgrouped as MW

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(rng, shape, choices=None):
    if choices is None:
        x = rng.standard_normal(shape).astype(np.float32)
    else:
        x = rng.choice(np.asarray(choices, dtype=np.float32), size=shape)
    return torch.from_numpy(x).to(torch.bfloat16)


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t):
    return t.to(torch.float64).numpy()


# ------------------------------------------------------------------------------------------
# Exact brute force
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["offsets", "indices", "masked"])
@pytest.mark.parametrize("b_major", ["k", "mn"])
def test_brute_force_fraction(layout, b_major):
    rng = np.random.default_rng(3)
    G, N, K = 3, 4, 6
    if layout == "offsets":
        groups, m = np.array([2, 2, 5]), 5            # group 1 empty
        rows = 5
    elif layout == "indices":
        groups, m = np.array([2, 0, 0, 2, 1]), 5      # unsorted ids
        rows = 5
    else:
        groups, m = np.array([1, 0, 3]), 3            # max_m = 3
        rows = G * m
    A = bf16(rng, (rows, K))
    Bs = bf16(rng, (G, N, K) if b_major == "k" else (G, K, N))
    D, S = MO.mgrouped_from_storage(bits(A), bits(Bs), layout, groups, m, b_major=b_major,
                                    d_init=np.zeros((rows, N)))
    Af = [[Fraction(float(v)) for v in row] for row in f64(A)]
    Bf = f64(Bs)
    owners = {}
    if layout == "offsets":
        prev = 0
        for g, end in enumerate(groups):
            for r in range(prev, end):
                owners[r] = g
            prev = end
    elif layout == "indices":
        owners = {r: int(g) for r, g in enumerate(groups)}
    else:
        for g in range(G):
            for j in range(groups[g]):
                owners[g * m + j] = g
    for r in range(rows):
        for n in range(N):
            if r not in owners:
                assert D[r, n] == 0.0 and S[r, n] == 0.0
                continue
            g = owners[r]
            w = [Fraction(float(Bf[g, n, kk] if b_major == "k" else Bf[g, kk, n])) for kk in range(K)]
            exact = sum(Af[r][kk] * w[kk] for kk in range(K))
            mag = sum(abs(Af[r][kk] * w[kk]) for kk in range(K))
            assert abs(Fraction(D[r, n]) - exact) <= Fraction(1, 10 ** 12) * (mag + 1)
            assert abs(Fraction(S[r, n]) - mag) <= Fraction(1, 10 ** 12) * (mag + 1)


# ------------------------------------------------------------------------------------------
# Special cases and closed forms
# ------------------------------------------------------------------------------------------

def test_single_group_is_plain_gemm():
    rng = np.random.default_rng(4)
    A, B = bf16(rng, (256, 64)), bf16(rng, (1, 128, 64))
    D, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", [256], 256, b_major="k")
    ref = torch.matmul(A.to(torch.float64), B[0].to(torch.float64).t()).numpy()
    assert np.allclose(D, ref, rtol=0, atol=1e-12)


def test_dgrad_orientation_is_plain_gemm():
    rng = np.random.default_rng(5)
    A, B = bf16(rng, (128, 96)), bf16(rng, (1, 96, 32))
    D, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", [128], 128, b_major="mn")
    ref = torch.matmul(A.to(torch.float64), B[0].to(torch.float64)).numpy()
    assert np.allclose(D, ref, rtol=0, atol=1e-12)


def test_ones_closed_form():
    G, N, K = 3, 8, 40
    groups = np.array([128, 128, 384])
    A = torch.ones(384, K, dtype=torch.bfloat16)
    B = torch.ones(G, N, K, dtype=torch.bfloat16)
    D, S = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", groups, 384)
    assert np.all(D == K) and np.all(S == K)


def test_group_picks_its_own_weight():
    """B_g = g * ones: every row of group g equals g * sum(A[r])."""
    G, N, K = 4, 2, 16
    rng = np.random.default_rng(6)
    A = bf16(rng, (512, K), choices=[-1.0, 0.5, 2.0])
    B = torch.stack([torch.full((N, K), float(g), dtype=torch.bfloat16) for g in range(G)])
    groups = np.array([128, 128, 384, 512])
    D, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", groups, 512)
    rowsum = f64(A).sum(axis=1)
    owner = np.repeat([0, 1, 2, 3], [128, 0, 256, 128])
    assert np.array_equal(D, (owner * rowsum)[:, None].repeat(N, axis=1))


def test_k_major_and_n_major_storage_agree():
    rng = np.random.default_rng(7)
    A, Bk = bf16(rng, (384, 64)), bf16(rng, (3, 32, 64))
    Bn = Bk.transpose(1, 2).contiguous()
    groups = np.array([128, 128, 384])
    Dk, Sk = MO.mgrouped_from_storage(bits(A), bits(Bk), "offsets", groups, 384, b_major="k")
    Dn, Sn = MO.mgrouped_from_storage(bits(A), bits(Bn), "offsets", groups, 384, b_major="mn")
    assert np.array_equal(Dk, Dn) and np.array_equal(Sk, Sn)


# ------------------------------------------------------------------------------------------
# Layout equivalences and masked semantics
# ------------------------------------------------------------------------------------------

def test_offsets_and_indices_layouts_agree():
    rng = np.random.default_rng(8)
    counts = np.array([256, 0, 128, 384])
    A, B = bf16(rng, (768, 32)), bf16(rng, (4, 16, 32))
    offs = np.cumsum(counts)
    ids = np.repeat(np.arange(4), counts)
    D1, S1 = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", offs, 768)
    D2, S2 = MO.mgrouped_from_storage(bits(A), bits(B), "indices", ids, 768)
    assert np.array_equal(D1, D2) and np.array_equal(S1, S2)


def test_shuffled_blocks_permute_rows():
    """Index layout: moving a 128-row block (its A rows and its id together) moves its D rows."""
    rng = np.random.default_rng(9)
    A, B = bf16(rng, (512, 32)), bf16(rng, (3, 16, 32))
    ids = np.repeat([0, 2, 2, 1], 128)
    perm = np.array([2, 0, 3, 1])
    rows = (perm[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    D1, _ = MO.mgrouped_from_storage(bits(A), bits(B), "indices", ids, 512)
    D2, _ = MO.mgrouped_from_storage(bits(A[rows]), bits(B), "indices", ids[rows], 512)
    assert np.array_equal(D1[rows], D2)


def test_masked_equals_contiguous_on_valid_rows_and_keeps_the_rest():
    rng = np.random.default_rng(10)
    G, max_m, N, K = 3, 200, 16, 32
    masked_m = np.array([200, 0, 57])
    A, B = bf16(rng, (G, max_m, K)), bf16(rng, (G, N, K))
    d0 = rng.standard_normal((G * max_m, N))
    D, S = MO.mgrouped_from_storage(bits(A), bits(B), "masked", masked_m, max_m, d_init=d0)
    packed = torch.cat([A[g, :masked_m[g]] for g in range(G)])
    Dc, Sc = MO.mgrouped_from_storage(bits(packed), bits(B), "offsets", np.cumsum(masked_m), int(masked_m.sum()))
    own = MO.owned_mask("masked", masked_m, max_m, G, G * max_m)
    assert own.sum() == masked_m.sum()
    assert np.array_equal(D[own], Dc) and np.array_equal(S[own], Sc)
    assert np.array_equal(D[~own], d0[~own]), "rows past masked_m must keep their contents"
    assert np.all(S[~own] == 0)


def test_accumulate_is_previous_plus_overwrite():
    rng = np.random.default_rng(11)
    A, B = bf16(rng, (256, 32)), bf16(rng, (2, 16, 32))
    d0 = rng.standard_normal((256, 16))
    D0, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", [128, 256], 256)
    D1, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", [128, 256], 256, d_init=d0, accumulate=True)
    assert np.allclose(D1, d0 + D0, rtol=0, atol=1e-12)


def test_rows_are_independent():
    """Permuting rows inside one group permutes the output rows and nothing else."""
    rng = np.random.default_rng(12)
    A, B = bf16(rng, (256, 32)), bf16(rng, (2, 16, 32))
    perm = np.concatenate([rng.permutation(128), 128 + rng.permutation(128)])
    D1, _ = MO.mgrouped_from_storage(bits(A), bits(B), "offsets", [128, 256], 256)
    D2, _ = MO.mgrouped_from_storage(bits(A[perm]), bits(B), "offsets", [128, 256], 256)
    assert np.array_equal(D1[perm], D2)


# ------------------------------------------------------------------------------------------
# Forward / dgrad / wgrad of one layer (section 5): ties to the K-grouped oracle
# ------------------------------------------------------------------------------------------

def test_forward_dgrad_wgrad_inner_product_identity():
    """For Y_g = X_g W_g^T, dX_g = dY_g W_g and dW_g = dY_g^T X_g (section 5):
    <dY_g, Y_g> = <dW_g, W_g> = <dX_g, X_g>. The wgrad side comes from the K-grouped oracle,
    whose own pins are independent of this module; a transposed or misplaced operand on either
    side breaks the equality."""
    rng = np.random.default_rng(13)
    G, n_in, n_out = 3, 24, 40
    counts = np.array([256, 0, 128])
    M = int(counts.sum())
    X, dY = bf16(rng, (M, n_in)), bf16(rng, (M, n_out))
    Wt = bf16(rng, (G, n_out, n_in))        # W_g: [out, in], K-major for the forward
    offs = np.cumsum(counts)
    Y, _ = MO.mgrouped_from_storage(bits(X), bits(Wt), "offsets", offs, M, b_major="k")
    dX, _ = MO.mgrouped_from_storage(bits(dY), bits(Wt), "offsets", offs, M, b_major="mn")
    # K-grouped: A = dY^T [out, tokens] (K-major), B = X [tokens, in] (N-major)
    dW, _ = KO.wgrad_from_storage(bits(dY.t().contiguous()), bits(X), offs.astype(np.int32), n_out, n_in)
    Wf, Xf, dYf = f64(Wt), f64(X), f64(dY)
    prev = 0
    for g, end in enumerate(offs):
        lhs = float(np.sum(dYf[prev:end] * Y[prev:end]))
        mid = float(np.sum(dW[g] * Wf[g]))
        rhs = float(np.sum(dX[prev:end] * Xf[prev:end]))
        scale = 1e-10 * (1 + np.abs(dYf[prev:end]).sum() * np.abs(Wf[g]).sum() * (np.abs(Xf).max() + 1))
        assert abs(lhs - mid) <= scale and abs(rhs - mid) <= scale, (g, lhs, mid, rhs)
        prev = end


# ------------------------------------------------------------------------------------------
# Layout rules and the pages' example
# ------------------------------------------------------------------------------------------

def test_layout_rules():
    assert MO.layout_valid("offsets", [128, 128, 384], 384, 3)            # zero count allowed
    assert not MO.layout_valid("offsets", [128, 200, 384], 384, 3)        # not tile-aligned
    assert not MO.layout_valid("offsets", [256, 128, 384], 384, 3)        # decreasing
    assert not MO.layout_valid("offsets", [128, 256, 256], 384, 3)        # last != m
    ids = np.repeat([1, 0, 1], 128)
    assert MO.layout_valid("indices", ids, 384, 2)                         # unsorted blocks fine
    bad = ids.copy()
    bad[130] = 1
    assert not MO.layout_valid("indices", bad, 384, 2)                     # a block with two ids
    assert not MO.layout_valid("indices", np.full(384, 2), 384, 2)         # id out of range
    assert MO.layout_valid("masked", [0, 7, 300], 300, 3)
    assert not MO.layout_valid("masked", [0, 7, 301], 300, 3)
    assert not MO.layout_valid("masked", [-1, 7, 3], 300, 3)


def test_pages_m_indices_example():
    """The per-row group ids printed for the contiguous layout (section 2.1) assign rows 0-2 to
    group 0, rows 3-4 to group 1 and rows 5-8 to group 2."""
    path = os.path.join(GOLDEN, "mgrouped_m_indices_example.txt")
    lines = [l for l in open(path) if l.strip() and not l.startswith("#")]
    ids = np.array([int(v) for v in lines[0].split()])
    expect = {int(k): [int(v) for v in rest.split(",")] for k, rest in (l.split(":") for l in lines[1:])}
    got = MO.group_rows("indices", ids, len(ids), 3)
    assert {g: r.tolist() for g, r in enumerate(got)} == expect
    for r in range(len(ids)):
        assert MO.group_of_row("indices", ids, len(ids), r) == ids[r]


def test_group_of_row_all_layouts():
    offs = np.array([128, 128, 384])
    assert [MO.group_of_row("offsets", offs, 384, r) for r in (0, 127, 128, 383)] == [0, 0, 2, 2]
    mm = np.array([3, 0, 5])
    assert MO.group_of_row("masked", mm, 10, 2) == 0
    assert MO.group_of_row("masked", mm, 10, 3) == -1
    assert MO.group_of_row("masked", mm, 10, 10) == -1
    assert MO.group_of_row("masked", mm, 10, 24) == 2
    assert MO.group_of_row("masked", mm, 10, 25) == -1


@pytest.mark.parametrize("layout,b_major", [("offsets", "k"), ("indices", "mn"), ("masked", "k")])
def test_element_from_storage_matches_full(layout, b_major):
    rng = np.random.default_rng(14)
    G, N, K = 3, 16, 48
    if layout == "masked":
        groups, m, rows = np.array([100, 0, 128]), 128, 3 * 128
        A = bf16(rng, (G, m, K))
    elif layout == "indices":
        groups, m, rows = np.repeat([2, 0, 2], 128), 384, 384
        A = bf16(rng, (rows, K))
    else:
        groups, m, rows = np.array([128, 128, 384]), 384, 384
        A = bf16(rng, (rows, K))
    B = bf16(rng, (G, N, K) if b_major == "k" else (G, K, N))
    D, S = MO.mgrouped_from_storage(bits(A), bits(B), layout, groups, m, b_major=b_major,
                                    d_init=np.zeros((rows, N)))
    own = MO.owned_mask(layout, groups, m, G, rows)
    for r in np.nonzero(own)[0][::7]:
        for c in (0, 5, N - 1):
            v, s = MO.element_from_storage(bits(A), bits(B), layout, groups, m, int(r), c, b_major=b_major)
            assert abs(v - D[r, c]) <= 1e-12 * (1 + S[r, c]) and abs(s - S[r, c]) <= 1e-12 * (1 + S[r, c])


# ------------------------------------------------------------------------------------------
# Workload recipe
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", sorted(MW.MG_NAMED))
def test_named_workloads_follow_layout_rules(name):
    w = MW.MG_NAMED[name]()
    g = MW.groups_array(w)
    assert MO.layout_valid(w.layout, g, w.m, w.num_groups)
    assert w.n % 256 == 0 and w.k % 64 == 0
    if w.layout != "masked":
        assert np.all(np.asarray(w.counts) % 128 == 0)


def test_shuffled_index_workload_is_valid_and_seeded():
    w = MW.mg_custom(4, 256, 64, "indices", [256, 0, 384, 128], seed=3, shuffle_blocks=True)
    g1, g2 = MW.groups_array(w), MW.groups_array(w)
    assert np.array_equal(g1, g2) and MO.layout_valid("indices", g1, w.m, 4)
    assert sorted(np.bincount(g1, minlength=4).tolist()) == sorted([256, 0, 384, 128])


def test_mg_inputs_are_seeded():
    w = MW.mg_custom(2, 256, 64, "masked", [5, 77], seed=9, max_m=96)
    x1, x2 = MW.make_mg_inputs(w), MW.make_mg_inputs(w)
    assert torch.equal(x1.a, x2.a) and torch.equal(x1.b, x2.b) and torch.equal(x1.d0, x2.d0)
    assert x1.a.shape == (2, 96, 64) and x1.b.shape == (2, 256, 64) and x1.d0.shape == (2, 96, 256)


# ------------------------------------------------------------------------------------------
# FP8 (per-block 1x128 scaling along K, section 3)
# ------------------------------------------------------------------------------------------

def _u8(t):
    return t.contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("b_major", ["k", "mn"])
def test_fp8_unit_scales_equal_the_bf16_oracle(b_major):
    """With every scale 1 the FP8 result is the BF16-path oracle on the decoded e4m3 values (all
    of which are exact in bf16): ties FP8 decoding and layout to the pinned BF16 definition."""
    rng = np.random.default_rng(40)
    G, N, K = 3, 32, 256
    a8 = torch.from_numpy(rng.standard_normal((384, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    b_shape = (G, N, K) if b_major == "k" else (G, K, N)
    b8 = torch.from_numpy(rng.standard_normal(b_shape).astype(np.float32)).to(torch.float8_e4m3fn)
    sfa = np.ones((K // 128, 384), dtype=np.float32)
    sfb = np.ones((G, K // 128, N), dtype=np.float32)
    groups = np.array([128, 128, 384])
    D8, S8 = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), sfa, sfb, "offsets", groups, 384, b_major=b_major)
    D16, S16 = MO.mgrouped_from_storage(bits(a8.to(torch.bfloat16)), bits(b8.to(torch.bfloat16)), "offsets",
                                        groups, 384, b_major=b_major)
    assert np.array_equal(D8, D16) and np.array_equal(S8, S16)


def test_fp8_scale_blocks_scale_exactly():
    """Doubling the scale of one 128-K block of one row doubles exactly that block's contribution."""
    rng = np.random.default_rng(41)
    G, N, K = 2, 16, 256
    a8 = torch.from_numpy(rng.standard_normal((256, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    b8 = torch.from_numpy(rng.standard_normal((G, N, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    sfa = np.ones((2, 256), dtype=np.float32)
    sfb = np.ones((G, 2, N), dtype=np.float32)
    groups = np.array([128, 256])
    D0, _ = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), sfa, sfb, "offsets", groups, 256)
    sfa2 = sfa.copy()
    sfa2[1, 200] = 4.0                                  # row 200 (group 1), K block 1
    D1, _ = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), sfa2, sfb, "offsets", groups, 256)
    a = KO.e4m3_to_f64(_u8(a8)).reshape(a8.shape)
    b = KO.e4m3_to_f64(_u8(b8)).reshape(b8.shape)
    blk = a[200, 128:] @ b[1][:, 128:].T
    assert np.array_equal(np.delete(D1, 200, axis=0), np.delete(D0, 200, axis=0))
    assert np.allclose(D1[200] - D0[200], 3.0 * blk, rtol=0, atol=1e-9)
    sfb2 = sfb.copy()
    sfb2[0, 0, 5] = 0.5                                 # group 0, K block 0, column 5
    D2, _ = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), sfa, sfb2, "offsets", groups, 256)
    changed = np.nonzero(np.any(D2 != D0, axis=1))[0]
    assert changed.min() >= 0 and changed.max() < 128 and np.all(np.nonzero(np.any(D2 != D0, axis=0))[0] == 5)


def test_fp8_ue8m0_scales_match_the_f32_form():
    """Packed UE8M0 words whose four bytes are equal describe the same per-128 scale as FP32."""
    rng = np.random.default_rng(42)
    G, N, K = 2, 16, 256
    a8 = torch.from_numpy(rng.standard_normal((256, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    b8 = torch.from_numpy(rng.standard_normal((G, K, N)).astype(np.float32)).to(torch.float8_e4m3fn)
    ea = rng.integers(120, 134, size=(2, 256))
    eb = rng.integers(120, 134, size=(G, 2, N))
    pack = lambda e: (e.astype(np.uint32) * 0x01010101).view(np.int32)
    f32 = lambda e: np.ldexp(1.0, e - 127).astype(np.float32)
    groups = np.array([128, 256])
    Dp, _ = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), pack(ea), pack(eb), "offsets", groups, 256,
                                         b_major="mn", sf_format="ue8m0_32")
    Df, _ = MO.mgrouped_fp8_from_storage(_u8(a8), _u8(b8), f32(ea), f32(eb), "offsets", groups, 256,
                                         b_major="mn")
    assert np.array_equal(Dp, Df)


def test_fp8_element_matches_full():
    w = MW.mg_custom(3, 256, 256, "masked", [100, 0, 128], seed=43, max_m=128, fp8=True)
    x = MW.make_mg_inputs(w)
    D, S = MO.mgrouped_fp8_from_storage(_u8(x.a), _u8(x.b), x.sfa.numpy(), x.sfb.numpy(), "masked",
                                        x.groups.numpy(), 128, d_init=np.zeros((w.rows, w.n)))
    for (r, c) in [(0, 0), (99, 255), (256, 17), (383, 200)]:
        v, s = MO.element_fp8_from_storage(_u8(x.a), _u8(x.b), x.sfa.numpy(), x.sfb.numpy(), "masked",
                                           x.groups.numpy(), 128, r, c)
        assert abs(v - D[r, c]) <= 1e-12 * (1 + S[r, c])
