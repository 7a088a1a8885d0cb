"""CPU oracle for the M-grouped MoE GEMM (forward and dgrad of a grouped linear layer).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA
library: it decodes the stored operand bits itself and evaluates the
definition in float64 with numpy.

What it computes ("05 · Grouped GEMM 与 Expert 计算", sections 1, 2 and 5):
only the M dimension varies between groups; N and K are fixed. Row r of A
belongs to one group g and is multiplied by that group's weight B_g:

    forward  Y_i  = X_i @ W_i^T    B stored [G, N, K] ("nt", K contiguous)
    dgrad    dX_i = dY_i @ W_i     B stored [G, K, N] (N contiguous)

so D[r, :] = A[r, :] @ op(B_g) with op(B_g) = B_g^T for the first storage and
B_g for the second (section 5.1: the dgrad takes the weight untransposed).

Which rows belong to which group comes in one of three layouts (section 2):
  "offsets"  contiguous rows, group g owns [offsets[g-1], offsets[g])
  "indices"  contiguous rows, m_indices[r] is the group of row r (section 2.1)
  "masked"   A [G, max_m, K]: group g owns its first masked_m[g] rows; the
             remaining rows of D are not computed and keep their contents
             (section 2.2)
With accumulate the result is added to D's previous contents; otherwise it
replaces them. Alignment rules (every contiguous segment a multiple of 128
rows, section 2.1) are the caller's contract and are checked by
``layout_valid``; the arithmetic itself does not depend on them.

FP8 (section 3: per-block 1x128 scaling along K): every e4m3 element is
multiplied by its scale before the product; row r of A carries one scale per
128 consecutive K (sfa [K/128, rows], MN-major), and so does column n of each
group's weight (sfb [G, K/128, N]). Scales may also be packed UE8M0 words with
one byte per 32 K (the same format as the K-grouped FP8 path).
"""
from __future__ import annotations

import numpy as np

from .kgw_oracle import bf16_to_f64, decode_scales, e4m3_to_f64

MG_ALIGN = 128


def group_rows(layout: str, groups, m: int, num_groups: int):
    """Row indices of A/D (flattened to [rows, K] / [rows, N]) owned by each group.

    Returns a list of ``num_groups`` int64 arrays.
    """
    g = np.asarray(groups, dtype=np.int64).reshape(-1)
    if layout == "offsets":
        out, prev = [], 0
        for e in range(num_groups):
            out.append(np.arange(prev, int(g[e]), dtype=np.int64))
            prev = int(g[e])
        return out
    if layout == "indices":
        return [np.nonzero(g == e)[0].astype(np.int64) for e in range(num_groups)]
    if layout == "masked":
        return [e * m + np.arange(int(g[e]), dtype=np.int64) for e in range(num_groups)]
    raise ValueError(layout)


def layout_valid(layout: str, groups, m: int, num_groups: int) -> bool:
    """The layout rules of section 2: contiguous groups tile-aligned; masked counts within max_m."""
    g = np.asarray(groups, dtype=np.int64).reshape(-1)
    if layout == "offsets":
        if len(g) != num_groups:
            return False
        counts = np.diff(np.concatenate([[0], g]))
        return bool(np.all(counts >= 0) and np.all(counts % MG_ALIGN == 0) and int(g[-1]) == m)
    if layout == "indices":
        if len(g) != m or m % MG_ALIGN:
            return False
        if np.any(g < 0) or np.any(g >= num_groups):
            return False
        blocks = g.reshape(-1, MG_ALIGN) if m else g.reshape(0, MG_ALIGN)
        return bool(np.all(blocks == blocks[:, :1]))
    if layout == "masked":
        return bool(len(g) == num_groups and np.all(g >= 0) and np.all(g <= m))
    raise ValueError(layout)


def op_b(B: np.ndarray, b_major: str) -> np.ndarray:
    """op(B_g) as a [G, K, N] float64 array: B_g^T for K-major [G, N, K], B_g for N-major [G, K, N]."""
    return np.swapaxes(B, 1, 2) if b_major == "k" else B


def mgrouped(A: np.ndarray, B: np.ndarray, layout: str, groups, m: int, *, b_major: str = "k",
             d_init=None, accumulate: bool = False, with_bound: bool = True):
    """D in float64 and the magnitude sum S = |A| @ |op(B_g)| per owned row.

    A: float64 [rows, K] (masked: [G*max_m, K] flattened); B: float64 [G, N, K] or [G, K, N].
    d_init: D's previous contents [rows, N] (needed for accumulate and for rows no group owns);
    rows that no group owns are returned as d_init (NaN where d_init is None). S is zero there.
    """
    G = B.shape[0]
    opB = op_b(B, b_major)
    rows, K = A.shape
    N = opB.shape[2]
    assert opB.shape[1] == K
    D = np.full((rows, N), np.nan) if d_init is None else np.array(d_init, dtype=np.float64, copy=True)
    S = np.zeros((rows, N)) if with_bound else None
    for g, r in enumerate(group_rows(layout, groups, m, G)):
        if len(r) == 0:
            continue
        res = A[r] @ opB[g]
        D[r] = (D[r] + res) if accumulate else res
        if with_bound:
            S[r] = np.abs(A[r]) @ np.abs(opB[g])
    return D, S


def owned_mask(layout: str, groups, m: int, num_groups: int, rows: int) -> np.ndarray:
    """Boolean [rows]: the row belongs to some group (is computed and written)."""
    mask = np.zeros(rows, dtype=bool)
    for r in group_rows(layout, groups, m, num_groups):
        mask[r] = True
    return mask


def mgrouped_from_storage(a_bits, b_bits, layout: str, groups, m: int, *, b_major: str = "k",
                          d_init=None, accumulate: bool = False, with_bound: bool = True):
    """Decode stored BF16 operands (raw uint16 bits) and evaluate ``mgrouped``."""
    a = bf16_to_f64(a_bits)
    A = a.reshape(-1, a.shape[-1])
    B = bf16_to_f64(b_bits)
    return mgrouped(A, B, layout, groups, m, b_major=b_major, d_init=d_init, accumulate=accumulate,
                    with_bound=with_bound)


def dequantize_fp8(a_bits, b_bits, sfa, sfb, b_major: str = "k", sf_format: str = "f32_128"):
    """Decoded, scaled operands: A [rows, K] and B [G, N, K] (K-major) or [G, K, N] (N-major)."""
    a = e4m3_to_f64(a_bits)
    a = a.reshape(-1, np.asarray(a_bits).shape[-1])
    rows, K = a.shape
    sa, blk = decode_scales(sfa, sf_format)                     # [K/blk, rows]
    A = a * np.repeat(sa.T, blk, axis=1)
    b = e4m3_to_f64(b_bits).reshape(np.asarray(b_bits).shape)
    sfb = np.asarray(sfb)
    B = np.empty_like(b)
    for g in range(b.shape[0]):
        sb, _ = decode_scales(sfb[g], sf_format)                 # [K/blk, N]
        per_kn = np.repeat(sb, blk, axis=0)                      # [K, N]
        B[g] = b[g] * (per_kn.T if b_major == "k" else per_kn)
    return A, B


def mgrouped_fp8_from_storage(a_bits, b_bits, sfa, sfb, layout: str, groups, m: int, *, b_major: str = "k",
                              sf_format: str = "f32_128", d_init=None, accumulate: bool = False,
                              with_bound: bool = True):
    """Decode stored e4m3 operands and their scales, then evaluate ``mgrouped``."""
    A, B = dequantize_fp8(a_bits, b_bits, sfa, sfb, b_major, sf_format)
    return mgrouped(A, B, layout, groups, m, b_major=b_major, d_init=d_init, accumulate=accumulate,
                    with_bound=with_bound)


def element_fp8_from_storage(a_bits, b_bits, sfa, sfb, layout: str, groups, m: int, row: int, col: int, *,
                             b_major: str = "k", sf_format: str = "f32_128"):
    """(D[row, col] without accumulate, S[row, col]) from the stored FP8 operands and scales."""
    g = group_of_row(layout, groups, m, row)
    assert g >= 0, "row owned by no group"
    a = np.asarray(a_bits)
    K = a.shape[-1]
    sa, blk = decode_scales(sfa, sf_format)
    arow = e4m3_to_f64(a.reshape(-1, K)[row]) * np.repeat(sa[:, row], blk)
    b = np.asarray(b_bits)
    sb, _ = decode_scales(np.asarray(sfb)[g], sf_format)
    bcol = e4m3_to_f64(b[g, col, :] if b_major == "k" else b[g, :, col]) * np.repeat(sb[:, col], blk)
    return float(np.dot(arow, bcol)), float(np.dot(np.abs(arow), np.abs(bcol)))


def group_of_row(layout: str, groups, m: int, row: int) -> int:
    """The group that owns flattened row ``row`` (-1 if none)."""
    g = np.asarray(groups, dtype=np.int64).reshape(-1)
    if layout == "offsets":
        e = int(np.searchsorted(g, row, side="right"))
        return e if e < len(g) else -1
    if layout == "indices":
        return int(g[row])
    e, local = divmod(row, m)
    return e if local < int(g[e]) else -1


def element_from_storage(a_bits, b_bits, layout: str, groups, m: int, row: int, col: int, *,
                         b_major: str = "k"):
    """(D[row, col] without accumulate, S[row, col]) from the stored operands, for sampled checks.

    Only row ``row`` of A and column ``col`` of op(B_g) are decoded, so this works at full size.
    """
    g = group_of_row(layout, groups, m, row)
    assert g >= 0, "row owned by no group"
    a = np.asarray(a_bits)
    K = a.shape[-1]
    arow = bf16_to_f64(a.reshape(-1, K)[row])
    b = np.asarray(b_bits)
    bcol = bf16_to_f64(b[g, col, :] if b_major == "k" else b[g, :, col])
    return float(np.dot(arow, bcol)), float(np.dot(np.abs(arow), np.abs(bcol)))
