"""CPU oracle for the K-grouped MoE weight-gradient GEMM.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The product path (the CUDA library
and its Python binding) never imports, links or calls it, and this module
shares no code with it: it reads stored operand bits and does its own decoding
and arithmetic in float64 with numpy.

What it computes is the plain definition of the operation ("Grouped GEMM +
WGrad (Unified)", section "Operation"): for expert e, begin = 0 when e == 0,
else offsets[e-1]; end = offsets[e]; and

    Wgrad[e] = A[:, begin:end] @ B[begin:end, :]

with A [hidden, tokens_sum] and B [tokens_sum, intermediate]. In MoE terms this
is dW_e = dY_e^T X_e, a GEMM whose contraction axis is the per-expert token
count ("05 · Grouped GEMM 与 Expert 计算", section 5.2). With accumulate the
result is added to the existing output; without it the output is overwritten
and an empty expert yields zeros (section "Operation").

The FP8 variant multiplies every decoded e4m3 element by its per-128-token
FP32 scale before the product: a row m of A and a column n of B each carry one
scale per block of 128 consecutive tokens ("05 · Grouped GEMM 与 Expert 计算",
section 3: per-block 1x128 scaling, scales stored MN-major). The FP4 variant
does the same with e2m1 elements (two per byte along the token axis, first
token in the low nibble) and one UE8M0 scale per 32 tokens ("How to Use K-Grouped
GEMM ...", steps 1-2: FP4 casts with gran_k = 32 for both operands). Token
blocks start at each expert's first token (``token_scale_rows``); with the
pages' counts (multiples of 256) they are the global blocks k // 128.

Every product here is exact in float64 only up to rounding of the float64
sums; the tests pin it against exact rational brute force, so "the oracle"
means "the definition, evaluated in float64".
"""
from __future__ import annotations

import numpy as np

TOKEN_ALIGN = 256
SCALE_BLOCK = 128


# ---------------------------------------------------------------------------------------------
# Exact decoding of stored element bits
# ---------------------------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Decode raw bfloat16 bit patterns (uint16/int16) exactly to float64.

    A bfloat16 value is the upper half of an IEEE binary32 word, so shifting the
    16 bits up by 16 gives the binary32 word that holds the same value exactly.
    (BF16 contract: operands are torch.bfloat16.)
    """
    u = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_to_f64(bits) -> np.ndarray:
    """Decode raw float8 e4m3 (the 'fn' variant: no infinities) bit patterns to float64.

    Layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. Exponent field 0 is
    subnormal: m/8 * 2**-6. The pattern S.1111.111 is NaN; every other pattern with
    exponent field 15 is a normal number (max 448).
    """
    b = np.asarray(bits).view(np.uint8).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int64))
    sub = (m / 8.0) * 2.0 ** -6
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 15) & ((b & 0x7) == 7), np.nan, mag)
    return sign * mag


E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_to_f64(packed) -> np.ndarray:
    """Decode packed FP4 e2m1 bytes to float64, two elements per byte, low nibble first.

    A 4-bit code is 1 sign bit, 2 exponent bits (bias 1) and 1 mantissa bit: exponent field 0
    is subnormal m * 0.5, otherwise (1 + m/2) * 2**(e-1); there is no NaN or infinity, the
    largest magnitude is 6. The result has twice the elements of ``packed`` (flattened).
    """
    b = np.asarray(packed).view(np.uint8).reshape(-1).astype(np.int64)
    codes = np.empty(2 * b.size, dtype=np.int64)
    codes[0::2] = b & 0xF
    codes[1::2] = b >> 4
    e = (codes >> 1) & 0x3
    m = (codes & 0x1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, (1.0 + m / 2.0) * np.ldexp(1.0, (e - 1).astype(np.int64)))
    return np.where(codes & 0x8, -mag, mag)


# ---------------------------------------------------------------------------------------------
# Offsets (section "BF16 contract": non-decreasing cumulative sum, counts % 256 == 0,
# final offset == tokens_sum)
# ---------------------------------------------------------------------------------------------

def expert_ranges(offsets):
    """[(begin_e, end_e)] with begin_0 = 0 and begin_e = offsets[e-1] (section "Operation")."""
    off = [int(v) for v in np.asarray(offsets).tolist()]
    return [((0 if e == 0 else off[e - 1]), off[e]) for e in range(len(off))]


def offsets_valid(offsets, tokens_sum: int, align: int = TOKEN_ALIGN) -> bool:
    """The offsets contract: non-decreasing, every count a multiple of ``align`` (the pages' 256
    by default; the unaligned entry point relaxes it), last offset == tokens_sum."""
    off = [int(v) for v in np.asarray(offsets).tolist()]
    if len(off) == 0:
        return False
    prev = 0
    for v in off:
        n = v - prev
        if n < 0 or n % align != 0:
            return False
        prev = v
    return prev == tokens_sum


# ---------------------------------------------------------------------------------------------
# Logical operands from stored operands (section "BF16 contract", input_order)
# ---------------------------------------------------------------------------------------------

def logical_a(a_values: np.ndarray, hidden: int, offsets, input_order: str, a_major: str = "k") -> np.ndarray:
    """Logical A [hidden, tokens_sum] from its stored values ("Grouped GEMM + WGrad (Unified)",
    section "BF16 contract": A is (hidden, tokens_sum) with stride (tokens_sum, 1) K-major or
    (1, hidden) M-major; input_order "tensor_ragged" keeps only the unit-stride axis).

    K-major tensor2d: stored [hidden, tokens_sum]. K-major ragged: expert e's block is
    [hidden, n_e] row-major starting at element begin_e*hidden. M-major (either order): stored
    [tokens_sum, hidden]; expert e's rows are its [n_e, hidden] block, which already starts at
    element begin_e*hidden.
    """
    ranges = expert_ranges(offsets)
    tokens_sum = ranges[-1][1] if ranges else 0
    flat = np.asarray(a_values).reshape(-1)
    if a_major == "mn":
        return flat.reshape(tokens_sum, hidden).T
    if input_order == "tensor2d":
        return flat.reshape(hidden, tokens_sum)
    assert input_order == "ragged"
    out = np.zeros((hidden, tokens_sum), dtype=flat.dtype)
    for (b, e) in ranges:
        n = e - b
        if n:
            out[:, b:e] = flat[b * hidden:(b + n) * hidden].reshape(hidden, n)
    return out


def logical_b(b_values: np.ndarray, intermediate: int, offsets, input_order: str, b_major: str = "mn") -> np.ndarray:
    """Logical B [tokens_sum, intermediate] (section "BF16 contract": stride (intermediate, 1)
    N-major or (1, tokens_sum) K-major).

    N-major (either order): stored [tokens_sum, intermediate]; expert e's block [n_e, I] starts at
    element begin_e*I. K-major tensor2d: stored [intermediate, tokens_sum]. K-major ragged:
    expert e's block is [intermediate, n_e] row-major starting at element begin_e*intermediate.
    """
    ranges = expert_ranges(offsets)
    tokens_sum = ranges[-1][1] if ranges else 0
    flat = np.asarray(b_values).reshape(-1)
    if b_major == "mn":
        return flat.reshape(tokens_sum, intermediate)
    if input_order == "tensor2d":
        return flat.reshape(intermediate, tokens_sum).T
    out = np.zeros((tokens_sum, intermediate), dtype=flat.dtype)
    for (b, e) in ranges:
        n = e - b
        if n:
            out[b:e, :] = flat[b * intermediate:(b + n) * intermediate].reshape(intermediate, n).T
    return out


def unpack_ue8m0_32(packed) -> np.ndarray:
    """Packed UE8M0 words [tokens/128, other] -> float64 scales [tokens/32, other].

    Byte j (least significant first) of word [kb][r] is the biased exponent e of the scale
    2**(e - 127) of tokens 128*kb + 32*j .. +32 ("05 · Grouped GEMM 与 Expert 计算", section 3:
    UE8M0 scale format; "How to Use K-Grouped GEMM ...", step 2: gran_k = 32, packed UE8M0).
    """
    w = np.asarray(packed).view(np.uint32)
    nb, other = w.shape
    out = np.empty((nb * 4, other), dtype=np.float64)
    for j in range(4):
        e = ((w >> (8 * j)) & 0xFF).astype(np.int64)
        out[j::4, :] = np.ldexp(1.0, e - 127)
    return out


def token_scale_rows(offsets, block: int) -> np.ndarray:
    """Scale row of every token: int64 [tokens_sum].

    Each expert's tokens are cut into blocks of 128 from its own first token, the last block
    possibly partial (the pages pad every expert to the quantisation alignment before FP8/FP4
    casts, "05 · Grouped GEMM 与 Expert 计算", section 4: quantization padding of each expert
    segment); expert e's 128-token blocks take scale rows sb_e, sb_e + 1, ... with
    sb_e = sum over f < e of ceil(n_f / 128). A scale of ``block`` (128, or 32 for UE8M0
    sub-blocks) tokens is row sb_e * (128 / block) + (k - begin_e) // block. When every count is a
    multiple of 128 this is k // block: the global blocks of the aligned contract.
    """
    per = SCALE_BLOCK // block
    rows = []
    sb = 0
    for (b, end) in expert_ranges(offsets):
        n = end - b
        rows.append(sb * per + np.arange(n, dtype=np.int64) // block)
        sb += (n + SCALE_BLOCK - 1) // SCALE_BLOCK
    return np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)


def ue4m3_to_f64(bits) -> np.ndarray:
    """Decode unsigned E4M3 scale bytes (UE4M3: the e4m3 'fn' encoding without a sign bit) exactly.

    4 exponent bits (bias 7) and 3 mantissa bits: exponent field 0 is subnormal m/8 * 2**-6,
    otherwise (1 + m/8) * 2**(e-7); 0x7F (all ones) is NaN. A byte with bit 7 set is not a UE4M3
    value and decodes to NaN as well.
    """
    b = np.asarray(bits).view(np.uint8).astype(np.int64)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    v = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int64)))
    return np.where(((b & 0x7F) == 0x7F) | (b >= 0x80), np.nan, v)


def unpack_ue4m3_16(packed) -> np.ndarray:
    """Packed UE4M3 words [tokens/64, other] -> float64 scales [tokens/16, other].

    Byte j (least significant first) of word [w][r] scales tokens 64*w + 16*j .. +16 of row or
    column r: one scale per 16 tokens, the block size the cuDNN page's block-scaled contract
    defaults to (sf_vec_size = 16), in the unsigned E4M3 format of NVFP4 block scales.
    """
    w = np.asarray(packed).view(np.uint32)
    nw, other = w.shape
    out = np.empty((nw * 4, other), dtype=np.float64)
    for j in range(4):
        out[j::4, :] = ue4m3_to_f64(((w >> (8 * j)) & 0xFF).astype(np.uint8))
    return out


def apply_scales_rows(x: np.ndarray, scales: np.ndarray, block: int, rows=None) -> np.ndarray:
    """x [rows, tokens] * s[r(k), m] for scales [blocks, rows]; r(k) = k // block, or the given
    per-token scale rows (``token_scale_rows``)."""
    s = np.asarray(scales, dtype=np.float64)
    if rows is None:
        return x * np.repeat(s.T, block, axis=1)
    return x * s[np.asarray(rows), :].T


def apply_scales_cols(x: np.ndarray, scales: np.ndarray, block: int, rows=None) -> np.ndarray:
    """x [tokens, cols] * s[r(k), n] for scales [blocks, cols]; r(k) as in ``apply_scales_rows``."""
    s = np.asarray(scales, dtype=np.float64)
    if rows is None:
        return x * np.repeat(s, block, axis=0)
    return x * s[np.asarray(rows), :]


def decode_scales(sf, sf_format: str):
    """(scales as float64 [tokens/block, other], block) for each scale format: FP32 per 128 tokens,
    packed UE8M0 per 32 tokens, packed UE4M3 per 16 tokens."""
    if sf_format == "ue8m0_32":
        return unpack_ue8m0_32(sf), 32
    if sf_format == "ue4m3_16":
        return unpack_ue4m3_16(sf), 16
    # FP32 scales per 128 tokens ("f32_128": powers of two; "f32_any": any finite value)
    return np.asarray(sf, dtype=np.float64), SCALE_BLOCK


def global_factor(global_scale_a=None, global_scale_b=None) -> float:
    """The product of the per-tensor global scales (1 where one is not given), exactly as float64."""
    ga = 1.0 if global_scale_a is None else float(np.float32(global_scale_a))
    gb = 1.0 if global_scale_b is None else float(np.float32(global_scale_b))
    return ga * gb


# ---------------------------------------------------------------------------------------------
# The operation
# ---------------------------------------------------------------------------------------------

def wgrad(A: np.ndarray, B: np.ndarray, offsets, c_init=None, accumulate: bool = False,
          with_bound: bool = True):
    """Per-expert Wgrad in float64 ("Grouped GEMM + WGrad (Unified)", section "Operation").

    A: float64 [hidden, tokens_sum]; B: float64 [tokens_sum, intermediate].
    Returns (out, S): out [E, hidden, intermediate] is R_e (overwrite; zeros for an empty
    expert) or C_e + R_e (accumulate; C_e unchanged for an empty expert); S = |A_e| @ |B_e|
    is the magnitude sum used by the error bound (None when with_bound is False).
    """
    ranges = expert_ranges(offsets)
    E = len(ranges)
    H, T = A.shape
    T2, I = B.shape
    assert T == T2 == (ranges[-1][1] if ranges else 0)
    out = np.zeros((E, H, I), dtype=np.float64)
    S = np.zeros((E, H, I), dtype=np.float64) if with_bound else None
    for e, (b, end) in enumerate(ranges):
        if accumulate:
            out[e] = np.asarray(c_init[e], dtype=np.float64)
        if end > b:
            Ae, Be = A[:, b:end], B[b:end, :]
            out[e] += Ae @ Be
            if with_bound:
                S[e] = np.abs(Ae) @ np.abs(Be)
    return out, S


def wgrad_from_storage(a_bits, b_bits, offsets, hidden: int, intermediate: int, *,
                       input_order: str = "tensor2d", fp8: bool = False, sfa=None, sfb=None,
                       c_init=None, accumulate: bool = False, with_bound: bool = True,
                       a_major: str = "k", b_major: str = "mn", sf_format: str = "f32_128",
                       fp4: bool = False, global_scale_a=None, global_scale_b=None):
    """Decode stored operands (raw bits) and evaluate the operation in float64.

    a_bits/b_bits: uint16 (bf16), uint8 (e4m3) or uint8 packed e2m1 (fp4, K-major only) numpy
    arrays as stored. sfa [tokens/128, hidden], sfb [tokens/128, intermediate]: float32 scales
    or packed UE8M0 words (FP8/FP4). c_init: the pre-filled output values (any float dtype,
    decoded by the caller) or None.
    """
    if fp4:
        assert a_major == "k" and b_major == "k" and sf_format in ("ue8m0_32", "ue4m3_16")
        fp8 = True   # from here on the same steps: decoded elements times their scales
    dec = e2m1_to_f64 if fp4 else (e4m3_to_f64 if fp8 else bf16_to_f64)
    A = logical_a(dec(a_bits), hidden, offsets, input_order, a_major)
    B = logical_b(dec(b_bits), intermediate, offsets, input_order, b_major)
    if fp8:
        sa, blk = decode_scales(sfa, sf_format)
        sb, _ = decode_scales(sfb, sf_format)
        rows = token_scale_rows(offsets, blk)
        A = apply_scales_rows(A, sa, blk, rows)
        B = apply_scales_cols(B, sb, blk, rows)
    g = global_factor(global_scale_a, global_scale_b)
    if g != 1.0:
        # per-tensor global scales multiply the whole product (cuDNN page, "Block-scaled contract":
        # global_scale_a / global_scale_b where the low-precision format requires them)
        A = A * g
    return wgrad(A, B, offsets, c_init=c_init, accumulate=accumulate, with_bound=with_bound)


def wgrad_element(A: np.ndarray, B: np.ndarray, offsets, e: int, m: int, n: int):
    """One output element R_e[m, n] and its bound S_e[m, n] (for sampled checks at full size)."""
    b, end = expert_ranges(offsets)[e]
    a = A[m, b:end]
    bb = B[b:end, n]
    return float(np.dot(a, bb)), float(np.dot(np.abs(a), np.abs(bb)))


# ---------------------------------------------------------------------------------------------
# Tolerance
# ---------------------------------------------------------------------------------------------

def tolerance(S: np.ndarray, ref: np.ndarray, out_dtype: str, c_init=None) -> np.ndarray:
    """Per-element error bound for a GPU result against the float64 oracle.

    FP32 output: 2e-5*S + 1e-6 (FP32 accumulation over the ragged token axis).
    Accumulate into FP32 adds one FP32 rounding of the sum: 2**-23*(|C| + |ref|).
    BF16 output adds one final BF16 rounding: 2**-8*|ref|; FP16 output one FP16 rounding:
    2**-10*|ref| plus 2**-24 for the subnormal range.
    """
    tol = 2e-5 * S + 1e-6
    if c_init is not None:
        tol = tol + 2.0 ** -23 * (np.abs(np.asarray(c_init, dtype=np.float64)) + np.abs(ref))
    if out_dtype == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(ref)
    elif out_dtype == "f16":
        tol = tol + 2.0 ** -10 * np.abs(ref) + 2.0 ** -24
    return tol


def element_from_storage(a_bits, b_bits, offsets, hidden: int, intermediate: int, e: int, m: int, n: int, *,
                         input_order: str = "tensor2d", fp8: bool = False, sfa=None, sfb=None,
                         a_major: str = "k", b_major: str = "mn", sf_format: str = "f32_128",
                         fp4: bool = False):
    """R_e[m, n] and S_e[m, n] read straight from the stored operands (for sampled checks).

    Only row m of A_e and column n of B_e are decoded, so this works at full problem size.
    Addressing follows ``logical_a``/``logical_b``; FP8 scales follow
    ``apply_scales_rows``/``apply_scales_cols``.
    """
    b, end = expert_ranges(offsets)[e]
    cnt = end - b
    if cnt == 0:
        return 0.0, 0.0
    tokens_sum = expert_ranges(offsets)[-1][1]
    if fp4:
        # K-major only: a row of A / column of B is a contiguous element range [s, e) with s and e
        # even, i.e. the packed bytes [s/2, e/2)
        assert a_major == "k" and b_major == "k"
        fa, fb = np.asarray(a_bits).reshape(-1), np.asarray(b_bits).reshape(-1)
        if input_order == "tensor2d":
            sa0, sb0 = m * tokens_sum + b, n * tokens_sum + b
        else:
            sa0, sb0 = b * hidden + m * cnt, b * intermediate + n * cnt
        arow = e2m1_to_f64(fa[sa0 // 2:(sa0 + cnt) // 2])
        bcol = e2m1_to_f64(fb[sb0 // 2:(sb0 + cnt) // 2])
        sa, blk = decode_scales(sfa, sf_format)
        sb, _ = decode_scales(sfb, sf_format)
        ks = token_scale_rows(offsets, blk)[b:end]
        arow = arow * sa[ks, m]
        bcol = bcol * sb[ks, n]
        return float(np.dot(arow, bcol)), float(np.dot(np.abs(arow), np.abs(bcol)))
    dec = e4m3_to_f64 if fp8 else bf16_to_f64
    flat_a = np.asarray(a_bits).reshape(-1)
    if a_major == "mn":
        arow = dec(flat_a[b * hidden + m: end * hidden: hidden])
    elif input_order == "tensor2d":
        arow = dec(flat_a[m * tokens_sum + b: m * tokens_sum + end])
    else:
        arow = dec(flat_a[b * hidden + m * cnt: b * hidden + (m + 1) * cnt])
    flat_b = np.asarray(b_bits).reshape(-1)
    if b_major == "mn":
        bcol = dec(flat_b[b * intermediate + n: end * intermediate: intermediate])
    elif input_order == "tensor2d":
        bcol = dec(flat_b[n * tokens_sum + b: n * tokens_sum + end])
    else:
        bcol = dec(flat_b[b * intermediate + n * cnt: b * intermediate + (n + 1) * cnt])
    if fp8:
        sa, blk = decode_scales(sfa, sf_format)
        sb, _ = decode_scales(sfb, sf_format)
        ks = token_scale_rows(offsets, blk)[b:end]
        arow = arow * sa[ks, m]
        bcol = bcol * sb[ks, n]
    return float(np.dot(arow, bcol)), float(np.dot(np.abs(arow), np.abs(bcol)))


def expert_from_storage(a_bits, b_bits, offsets, hidden: int, intermediate: int, e: int, *,
                        input_order: str = "tensor2d", fp8: bool = False, sfa=None, sfb=None,
                        a_major: str = "k", b_major: str = "mn", sf_format: str = "f32_128",
                        fp4: bool = False, global_scale_a=None, global_scale_b=None):
    """(R_e, S_e) of one expert, decoding only that expert's operands (full-size checks).

    The same definition as ``wgrad_from_storage`` restricted to expert e: A_e [hidden, n_e] and
    B_e [n_e, intermediate] are read through the addressing of ``logical_a``/``logical_b``, each
    element multiplied by the scale of its token block (FP8/FP4, as in ``apply_scales_rows``/
    ``apply_scales_cols``), then R_e = A_e @ B_e and S_e = |A_e| @ |B_e| in float64. Memory is
    bounded by one expert's operands, so every output element of a full-size problem can be
    checked expert by expert. An empty expert gives zeros.
    """
    b, end = expert_ranges(offsets)[e]
    n = end - b
    if n == 0:
        z = np.zeros((hidden, intermediate), dtype=np.float64)
        return z, z.copy()
    tokens_sum = expert_ranges(offsets)[-1][1]
    fa = np.asarray(a_bits).reshape(-1)
    fb = np.asarray(b_bits).reshape(-1)
    if fp4:
        # packed e2m1, both operands K-major: tensor2d rows hold tokens_sum/2 bytes; ragged blocks
        # are [rows, n_e/2] bytes starting at byte begin_e*rows/2
        assert a_major == "k" and b_major == "k" and b % 2 == 0 and n % 2 == 0
        if input_order == "tensor2d":
            pa = fa.reshape(hidden, tokens_sum // 2)[:, b // 2:end // 2]
            pb = fb.reshape(intermediate, tokens_sum // 2)[:, b // 2:end // 2]
        else:
            pa = fa[b * hidden // 2:end * hidden // 2]
            pb = fb[b * intermediate // 2:end * intermediate // 2]
        Ae = e2m1_to_f64(np.ascontiguousarray(pa)).reshape(hidden, n)
        Be = e2m1_to_f64(np.ascontiguousarray(pb)).reshape(intermediate, n).T
    else:
        dec = e4m3_to_f64 if fp8 else bf16_to_f64
        if a_major == "mn":
            Ae = dec(fa[b * hidden:end * hidden]).reshape(n, hidden).T
        elif input_order == "tensor2d":
            Ae = dec(fa.reshape(hidden, tokens_sum)[:, b:end])
        else:
            Ae = dec(fa[b * hidden:end * hidden]).reshape(hidden, n)
        if b_major == "mn":
            Be = dec(fb[b * intermediate:end * intermediate]).reshape(n, intermediate)
        elif input_order == "tensor2d":
            Be = dec(fb.reshape(intermediate, tokens_sum)[:, b:end]).T
        else:
            Be = dec(fb[b * intermediate:end * intermediate]).reshape(intermediate, n).T
    if fp8 or fp4:
        sa, blk = decode_scales(sfa, sf_format)
        sb, _ = decode_scales(sfb, sf_format)
        ks = token_scale_rows(offsets, blk)[b:end]
        Ae = Ae * sa[ks, :].T
        Be = Be * sb[ks, :]
    g = global_factor(global_scale_a, global_scale_b)
    if g != 1.0:
        Ae = Ae * g
    return Ae @ Be, np.abs(Ae) @ np.abs(Be)
