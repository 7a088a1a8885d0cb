"""Seeded synthetic inputs for the K-grouped MoE weight-gradient GEMM.

This module only draws inputs. It holds none of the method's arithmetic
(no products, no sums over tokens, no scaling of products) so that both the
CUDA path and the CPU oracle can consume the same tensors without sharing
any computation.

Workloads follow the shapes of the pages' operation ("Grouped GEMM + WGrad
(Unified)", sections "Operation" and "BF16 contract"): A is
[hidden, tokens_sum] (K-major: stride (tokens_sum, 1)), B is
[tokens_sum, intermediate] (N-major: stride (intermediate, 1)), offsets is
the int32 cumulative token count per expert, and every per-expert count is a
multiple of 256. The per-expert counts of the balanced workloads use the
uniform(0.7, 1.3) spread of DeepGEMM's m-grouped generator described in
"05 · Grouped GEMM 与 Expert 计算", section 2.1.

Randomness: counts come from ``numpy.random.default_rng(seed)`` (draw order:
counts, then the choice of zeroed experts, then the expert permutation);
tensors come from a CPU ``torch.Generator`` seeded with ``seed`` (draw order:
A, B, then the pre-filled output C).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

TOKEN_ALIGN = 256  # every per-expert count is a multiple of 256 (BF16 contract)
FP8_BLOCK = 128    # one scale per 128 consecutive tokens, per row / column
E4M3_MAX = 448.0


def round_to_256(x: np.ndarray) -> np.ndarray:
    """Nearest multiple of 256: 256 * floor(x / 256 + 0.5)."""
    return (TOKEN_ALIGN * np.floor(np.asarray(x, dtype=np.float64) / TOKEN_ALIGN + 0.5)).astype(np.int64)


def counts_uniform_spread(seed: int, num_experts: int, mean_tokens: int, lo: float, hi: float,
                          zero_experts: int = 0) -> np.ndarray:
    """Per-expert counts round_to_256(mean * U(lo, hi)); optionally zero some experts."""
    rng = np.random.default_rng(seed)
    counts = round_to_256(mean_tokens * rng.uniform(lo, hi, size=num_experts))
    if zero_experts:
        zeroed = rng.choice(num_experts, size=zero_experts, replace=False)
        counts[zeroed] = 0
    return counts


def counts_zipf(seed: int, num_experts: int, total_tokens: int, s: float) -> np.ndarray:
    """Zipf(s) split of ``total_tokens`` over a random expert permutation.

    Rank r (1-based) gets weight r**-s; counts are 256*floor(total*p_r/256);
    the rounding deficit goes to rank 1 so the counts sum to ``total_tokens``
    exactly. A seeded permutation maps ranks to experts.
    """
    rng = np.random.default_rng(seed)
    r = np.arange(1, num_experts + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    by_rank = TOKEN_ALIGN * np.floor(total_tokens * p / TOKEN_ALIGN).astype(np.int64)
    by_rank[0] += total_tokens - int(by_rank.sum())
    perm = rng.permutation(num_experts)
    counts = np.zeros(num_experts, dtype=np.int64)
    counts[perm] = by_rank
    return counts


def offsets_from_counts(counts) -> np.ndarray:
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


@dataclasses.dataclass
class Workload:
    """Description of one synthetic problem (shapes, modes and the input recipe)."""
    name: str
    num_experts: int
    hidden: int
    intermediate: int
    counts: np.ndarray
    seed: int
    a_std: float = 1.0
    b_std: float = 1.0
    out_dtype: str = "f32"          # "f32" | "bf16" | "f16"
    accumulate: bool = False
    c_std: float = 1.0              # pre-filled output ~ N(0, c_std) when accumulating
    input_order: str = "tensor2d"   # "tensor2d" | "ragged"
    output_mode: str = "dense"      # "dense" | "discrete"
    fp8: bool = False
    a_major: str = "k"              # "k": A stored [hidden, tokens]; "mn": stored [tokens, hidden]
    sf_format: str = "f32_128"      # FP8 scales: "f32_128" (FP32 powers of two per 128 tokens) | "f32_any"
                                    # (general FP32 per 128 tokens) | "ue8m0_32" (packed) | "ue4m3_16" (NVFP4)
    b_major: str = "mn"             # "mn": B stored [tokens, intermediate]; "k": stored [intermediate, tokens]
    fp4: bool = False               # e2m1 operands (K-major A and B), UE8M0 scales per 32 tokens
    unaligned: bool = False         # counts multiples of 8, not 256 (the unaligned BF16 entry point)

    @property
    def tokens_sum(self) -> int:
        return int(np.asarray(self.counts).sum())

    @property
    def offsets(self) -> np.ndarray:
        return offsets_from_counts(self.counts)

    @property
    def flops(self) -> int:
        return 2 * self.hidden * self.intermediate * self.tokens_sum


def tiny() -> Workload:
    return Workload("tiny BF16: E=4 hidden=128 intermediate=256 counts [256,512,0,768]",
                    4, 128, 256, np.array([256, 512, 0, 768]), seed=0)


def balanced() -> Workload:
    return Workload("BF16 balanced: E=8 hidden=4096 intermediate=2048, FP32 dense overwrite",
                    8, 4096, 2048, counts_uniform_spread(1, 8, 4096, 0.7, 1.3), seed=1,
                    a_std=1.0, b_std=0.02)


def wide() -> Workload:
    return Workload("BF16 wide-hidden: E=32 hidden=7168 intermediate=2048, BF16 dense accumulate",
                    32, 7168, 2048, counts_uniform_spread(2, 32, 2048, 0.5, 1.5, zero_experts=2), seed=2,
                    out_dtype="bf16", accumulate=True)


def fp8() -> Workload:
    return Workload("FP8 block-scaled: E=16 hidden=4096 intermediate=1536, BF16 dense overwrite",
                    16, 4096, 1536, counts_uniform_spread(3, 16, 4096, 0.7, 1.3), seed=3,
                    out_dtype="bf16", fp8=True)


def skewed() -> Workload:
    return Workload("skewed ragged: E=128 hidden=2048 intermediate=768 Zipf(1.2) over 262144 tokens, "
                    "discrete BF16 outputs",
                    128, 2048, 768, counts_zipf(4, 128, 262144, 1.2), seed=4,
                    out_dtype="bf16", input_order="ragged", output_mode="discrete")


def round_to_8(x: np.ndarray) -> np.ndarray:
    """Nearest multiple of 8: 8 * floor(x / 8 + 0.5)."""
    return (8 * np.floor(np.asarray(x, dtype=np.float64) / 8 + 0.5)).astype(np.int64)


def unaligned() -> Workload:
    """The balanced shape with counts rounded to 8 tokens instead of 256 (same seed and spread)."""
    rng = np.random.default_rng(1)
    counts = round_to_8(4096 * rng.uniform(0.7, 1.3, size=8))
    return Workload("BF16 unaligned counts: E=8 hidden=4096 intermediate=2048, counts multiples of 8, "
                    "FP32 dense overwrite", 8, 4096, 2048, counts, seed=9, a_std=1.0, b_std=0.02,
                    unaligned=True)


def fp4() -> Workload:
    return Workload("FP4 block-scaled: E=16 hidden=4096 intermediate=1536, e2m1 with UE8M0 per 32 tokens, "
                    "K-major A and B, BF16 dense overwrite",
                    16, 4096, 1536, counts_uniform_spread(3, 16, 4096, 0.7, 1.3), seed=8,
                    out_dtype="bf16", fp4=True, b_major="k", sf_format="ue8m0_32")


def fp8_fp32() -> Workload:
    """The FP8 workload with general FP32 scales (amax/448, not rounded to powers of two)."""
    return Workload("FP8 general FP32 scales: E=16 hidden=4096 intermediate=1536, scale amax/448 per 128 tokens, "
                    "BF16 dense overwrite", 16, 4096, 1536, counts_uniform_spread(3, 16, 4096, 0.7, 1.3), seed=14,
                    out_dtype="bf16", fp8=True, sf_format="f32_any")


def nvfp4() -> Workload:
    return Workload("NVFP4 block-scaled: E=16 hidden=4096 intermediate=1536, e2m1 with UE4M3 scales per 16 "
                    "tokens and FP32 global scales, K-major A and B, BF16 dense overwrite",
                    16, 4096, 1536, counts_uniform_spread(3, 16, 4096, 0.7, 1.3), seed=13,
                    out_dtype="bf16", fp4=True, b_major="k", sf_format="ue4m3_16")


def round_to(x: np.ndarray, m: int) -> np.ndarray:
    """Nearest multiple of m: m * floor(x / m + 0.5)."""
    return (m * np.floor(np.asarray(x, dtype=np.float64) / m + 0.5)).astype(np.int64)


def fp8_unaligned() -> Workload:
    """The FP8 workload's shape with counts rounded to 16 tokens (same seed and spread)."""
    rng = np.random.default_rng(3)
    counts = round_to(4096 * rng.uniform(0.7, 1.3, size=16), 16)
    return Workload("FP8 unaligned counts: E=16 hidden=4096 intermediate=1536, counts multiples of 16, "
                    "per-expert 128-token scale blocks, BF16 dense overwrite", 16, 4096, 1536, counts, seed=11,
                    out_dtype="bf16", fp8=True, unaligned=True)


def fp4_unaligned() -> Workload:
    """The FP4 workload's shape with counts rounded to 32 tokens (same seed and spread)."""
    rng = np.random.default_rng(3)
    counts = round_to(4096 * rng.uniform(0.7, 1.3, size=16), 32)
    return Workload("FP4 unaligned counts: E=16 hidden=4096 intermediate=1536, counts multiples of 32, "
                    "e2m1 with UE8M0 per 32 tokens of each expert's 128-token blocks, BF16 dense overwrite",
                    16, 4096, 1536, counts, seed=12, out_dtype="bf16", fp4=True, b_major="k",
                    sf_format="ue8m0_32", unaligned=True)


NAMED = {"tiny": tiny, "balanced": balanced, "wide": wide, "fp8": fp8, "skewed": skewed, "fp4": fp4,
         "unaligned": unaligned, "fp8_unaligned": fp8_unaligned, "fp4_unaligned": fp4_unaligned, "nvfp4": nvfp4,
         "fp8_fp32": fp8_fp32}


def custom(num_experts: int, hidden: int, intermediate: int, counts, seed: int, **kw) -> Workload:
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.shape == (num_experts,)
    return Workload(f"custom E={num_experts} H={hidden} I={intermediate}", num_experts, hidden,
                    intermediate, counts, seed, **kw)


# --------------------------------------------------------------------------------------------
# Tensors
# --------------------------------------------------------------------------------------------

@dataclasses.dataclass
class Inputs:
    """Stored operands. All tensors live on ``device``.

    a: tensor2d -> [hidden, tokens_sum] row-major; ragged -> flat buffer where expert e's
       block [hidden, n_e] (row-major, leading dimension n_e) starts at element begin_e*hidden.
    b: [tokens_sum, intermediate] row-major (identical in both input orders, because B's
       unit-stride axis is the intermediate axis).
    With a_major "mn" A is stored [tokens_sum, hidden] (expert blocks [n_e, hidden] back to back
    in both orders); with b_major "k" B is stored [intermediate, tokens_sum] (tensor2d) or as
    per-expert [intermediate, n_e] blocks (ragged).
    sfa/sfb (FP8/FP4): float32 [blocks, hidden] / [blocks, intermediate] with one row per 128-token
       block of each expert (tokens_sum/128 rows when every count is a multiple of 128), or with
       sf_format "ue8m0_32" int32 packed UE8M0 words of the same shapes.
    c: pre-filled output [E, hidden, intermediate] for accumulate mode, else None.
    gsa/gsb (NVFP4, sf_format "ue4m3_16"): float32 [1] per-tensor global scales.
    """
    a: torch.Tensor
    b: torch.Tensor
    offsets: torch.Tensor
    sfa: Optional[torch.Tensor] = None
    sfb: Optional[torch.Tensor] = None
    c: Optional[torch.Tensor] = None
    gsa: Optional[torch.Tensor] = None      # NVFP4: float32 [1] global scale of A (decode multiplier)
    gsb: Optional[torch.Tensor] = None      # NVFP4: float32 [1] global scale of B


def out_torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[name]


def _normal(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def pow2_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Exponent k with 2**k = 2**ceil(log2(amax/448)) (k = 0 where amax == 0), computed exactly."""
    v = np.asarray(amax, dtype=np.float64) / E4M3_MAX
    frac, ex = np.frexp(v)            # v = frac * 2**ex, frac in [0.5, 1)
    k = np.where(frac == 0.5, ex - 1, ex)
    return np.where(v == 0.0, 0, k).astype(np.int64)


def quantize_e4m3_blocks(x: torch.Tensor, token_axis: int):
    """Quantise ``x`` (float32 2-D) to e4m3 with one power-of-two FP32 scale per 128 tokens.

    Returns (q [same shape, float8_e4m3fn], scales float32 [tokens/128, other]).
    The scale is 2**ceil(log2(amax/448)), so |x/scale| <= 448 and nothing saturates.
    """
    assert x.dim() == 2 and x.dtype == torch.float32
    xt = x if token_axis == 1 else x.t()          # [other, tokens]
    other, tokens = xt.shape
    assert tokens % FP8_BLOCK == 0
    blocks = xt.reshape(other, tokens // FP8_BLOCK, FP8_BLOCK)
    amax = blocks.abs().amax(dim=2)               # [other, nblk]
    k = pow2_scale_exponent(amax.numpy())
    scale = torch.from_numpy(np.ldexp(np.ones_like(k, dtype=np.float64), k).astype(np.float32))
    q = (blocks / scale.unsqueeze(2)).to(torch.float8_e4m3fn).reshape(other, tokens)
    if token_axis == 0:
        q = q.t().contiguous()
    return q.contiguous(), scale.t().contiguous()   # scales as [nblk, other]


def quantize_e4m3_fp32_blocks(x: torch.Tensor, token_axis: int):
    """Quantise ``x`` (float32 2-D) to e4m3 with one general FP32 scale per 128 tokens: the scale is
    amax/448 in float32, raised by one ulp when the division would otherwise exceed 448 (1 for an
    all-zero block), so the scales are in general not powers of two. Same return layout as
    ``quantize_e4m3_blocks``."""
    assert x.dim() == 2 and x.dtype == torch.float32
    xt = x if token_axis == 1 else x.t()
    other, tokens = xt.shape
    assert tokens % FP8_BLOCK == 0
    blocks = xt.reshape(other, tokens // FP8_BLOCK, FP8_BLOCK)
    amax = blocks.abs().amax(dim=2).numpy().astype(np.float32)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    over = (amax / np.maximum(scale, np.float32(1e-30))) > np.float32(E4M3_MAX)
    scale = np.where(over, np.nextafter(scale, np.float32(np.inf)), scale).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    st = torch.from_numpy(scale)
    q = (blocks / st.unsqueeze(2)).to(torch.float8_e4m3fn).reshape(other, tokens)
    if token_axis == 0:
        q = q.t().contiguous()
    return q.contiguous(), st.t().contiguous()


def quantize_e4m3_ue8m0_32(x: torch.Tensor, token_axis: int):
    """Quantise ``x`` (float32 2-D) to e4m3 with one power-of-two scale per 32 tokens, returned as
    packed UE8M0 words: int32 [tokens/128, other], byte j of word [kb][r] = 127 + log2(scale) of
    tokens 128*kb + 32*j .. +32 of row/column r (scale = 2**ceil(log2(amax/448)), 1 for amax 0).
    """
    assert x.dim() == 2 and x.dtype == torch.float32
    xt = x if token_axis == 1 else x.t()
    other, tokens = xt.shape
    assert tokens % FP8_BLOCK == 0
    blocks = xt.reshape(other, tokens // 32, 32)
    amax = blocks.abs().amax(dim=2)                       # [other, tokens/32]
    k = pow2_scale_exponent(amax.numpy())
    scale = torch.from_numpy(np.ldexp(np.ones_like(k, dtype=np.float64), k).astype(np.float32))
    q = (blocks / scale.unsqueeze(2)).to(torch.float8_e4m3fn).reshape(other, tokens)
    if token_axis == 0:
        q = q.t().contiguous()
    byte = (k + 127).astype(np.uint32).reshape(other, tokens // 128, 4)
    words = (byte[..., 0] | (byte[..., 1] << 8) | (byte[..., 2] << 16) | (byte[..., 3] << 24)).astype(np.uint32)
    packed = torch.from_numpy(words.view(np.int32).T.copy())   # [tokens/128, other]
    return q.contiguous(), packed


E2M1_MAX = 6.0
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_codes(v: np.ndarray) -> np.ndarray:
    """Round float64 values with |v| <= 6 to the nearest e2m1 code (ties to the even code)."""
    a = np.abs(v)
    idx = np.searchsorted(_E2M1_GRID, a)                 # first grid point >= |v|
    idx = np.clip(idx, 1, 7)
    lo, hi = _E2M1_GRID[idx - 1], _E2M1_GRID[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((idx & 1) == 0))
    code = np.where(pick_hi, idx, idx - 1)
    code = np.where(a == 0.0, 0, code)
    return (code | np.where(np.signbit(v) & (code != 0), 8, 0)).astype(np.uint8)


_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_e2m1_ue8m0_32(x: torch.Tensor, token_axis: int):
    """Quantise ``x`` (float32 2-D) to FP4 e2m1 with one power-of-two scale per 32 tokens.

    Returns (packed uint8 [other, tokens/2]: the token axis contiguous, two elements per byte, the
    first in the low nibble; packed UE8M0 words int32 [tokens/128, other] as in
    ``quantize_e4m3_ue8m0_32``). The scale is 2**ceil(log2(amax/6)) (1 for amax 0), so
    |x/scale| <= 6 and nothing saturates; elements round to the nearest e2m1 value, ties to the
    even code (the same rule as ``e2m1_codes``).
    """
    assert x.dim() == 2 and x.dtype == torch.float32
    xt = (x if token_axis == 1 else x.t()).contiguous()
    other, tokens = xt.shape
    assert tokens % FP8_BLOCK == 0
    blocks = xt.view(other, tokens // 32, 32)
    amax = blocks.abs().amax(dim=2).double().numpy()
    v = amax / E2M1_MAX
    frac, ex = np.frexp(v)
    k = np.where(v == 0.0, 0, np.where(frac == 0.5, ex - 1, ex)).astype(np.int64)
    scale = torch.from_numpy(np.ldexp(1.0, k).astype(np.float32))
    mids = torch.tensor(_E2M1_MIDS, dtype=torch.float32)
    packed = torch.empty((other, tokens // 2), dtype=torch.uint8)
    step = max(1, (1 << 22) // tokens)
    for r0 in range(0, other, step):          # row chunks bound the temporaries
        y = blocks[r0:r0 + step] / scale[r0:r0 + step, :, None]    # exact: power-of-two scale
        a = y.abs().reshape(-1)
        code = torch.bucketize(a, mids)                              # ties land on the lower code
        tie_up = (code < 7) & (a == mids[code.clamp(max=6)]) & ((code & 1) == 1)
        code = code + tie_up.to(code.dtype)
        neg = torch.signbit(y.reshape(-1)) & (code != 0)
        code = (code | (neg.to(code.dtype) << 3)).to(torch.uint8).view(-1, tokens)
        packed[r0:r0 + step] = code[:, 0::2] | (code[:, 1::2] << 4)
    byte = (k + 127).astype(np.uint32).reshape(other, tokens // 128, 4)
    words = (byte[..., 0] | (byte[..., 1] << 8) | (byte[..., 2] << 16) | (byte[..., 3] << 24)).astype(np.uint32)
    return packed, torch.from_numpy(words.view(np.int32).T.copy())


def expert_padded_columns(counts):
    """(cols, width): the column of every token in the layout where each expert's block starts on a
    multiple of 128 (each expert padded to whole 128-token blocks, as the pages' quantization
    padding does before FP8/FP4 casts), and that layout's width (sum of ceil(n_e/128)*128)."""
    cols, start = [], 0
    for n in np.asarray(counts, dtype=np.int64).tolist():
        cols.append(start + np.arange(n, dtype=np.int64))
        start += -(-n // FP8_BLOCK) * FP8_BLOCK
    return (np.concatenate(cols) if cols else np.zeros(0, dtype=np.int64)), start


def quantize_per_expert(quantize, x: torch.Tensor, token_axis: int, counts, packed_fp4: bool = False):
    """Apply a block quantiser with each expert's tokens padded to whole 128-token blocks.

    The scales come out one row per 128-token block of each expert ([sum ceil(n_e/128), other]);
    the quantised operand keeps the unpadded token layout (padding zeros never change a block's
    amax). With counts that are multiples of 128 this is ``quantize`` itself. ``packed_fp4``:
    ``quantize`` returns e2m1 bytes [other, tokens/2] (counts must then be even).
    """
    counts = np.asarray(counts, dtype=np.int64)
    if np.all(counts % FP8_BLOCK == 0):
        return quantize(x, token_axis)
    cols, width = expert_padded_columns(counts)
    idx = torch.from_numpy(cols)
    if token_axis == 1:
        xp = x.new_zeros((x.shape[0], width))
        xp[:, idx] = x
    else:
        xp = x.new_zeros((width, x.shape[1]))
        xp[idx, :] = x
    q, sf = quantize(xp, token_axis)
    if packed_fp4:
        assert np.all(counts % 2 == 0)
        return q[:, torch.from_numpy(cols[0::2] // 2)].contiguous(), sf
    u = q.view(torch.uint8)            # gather the bytes (float8 tensors cannot be indexed on every torch)
    return (u[:, idx] if token_axis == 1 else u[idx, :]).contiguous().view(q.dtype), sf


_E4M3_POS = None


def e4m3_positive_values() -> np.ndarray:
    """The finite positive values of the e4m3 'fn' encoding (codes 1..126), ascending."""
    global _E4M3_POS
    if _E4M3_POS is None:
        codes = torch.arange(1, 127, dtype=torch.uint8)
        _E4M3_POS = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return _E4M3_POS


def quantize_e2m1_ue4m3_16(x: torch.Tensor, token_axis: int, gs: float):
    """Quantise ``x`` (float32 2-D) to NVFP4: e2m1 elements, one unsigned-E4M3 scale per 16 tokens,
    and the per-tensor global scale ``gs`` (a decode multiplier: value = e2m1 * block scale * gs).

    The block scale is the smallest E4M3 value >= amax / (6 * gs) (1 for an all-zero block), so
    |x / (scale * gs)| <= 6 up to the float32 rounding of the division and nothing saturates;
    elements round to the nearest e2m1 value, ties to the even code. Returns (packed uint8
    [other, tokens/2], the token axis contiguous, first token in the low nibble; int32 words
    [tokens/64, other], byte j of word [w][r] = the scale code of tokens 64w + 16j .. +16).
    """
    assert x.dim() == 2 and x.dtype == torch.float32
    xt = (x if token_axis == 1 else x.t()).contiguous()
    other, tokens = xt.shape
    assert tokens % 64 == 0
    blocks = xt.view(other, tokens // 16, 16)
    amax = blocks.abs().amax(dim=2).double().numpy()
    need = amax / (E2M1_MAX * gs)
    vals = e4m3_positive_values()
    idx = np.minimum(np.searchsorted(vals, need, side="left"), len(vals) - 1)
    scale = np.where(amax == 0.0, 1.0, vals[idx])                          # exact E4M3 values
    codes = torch.from_numpy(scale.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    div = torch.from_numpy((scale * gs).astype(np.float32))
    mids = torch.tensor(_E2M1_MIDS, dtype=torch.float32)
    packed = torch.empty((other, tokens // 2), dtype=torch.uint8)
    step = max(1, (1 << 22) // tokens)
    for r0 in range(0, other, step):
        y = blocks[r0:r0 + step] / div[r0:r0 + step, :, None]
        a = y.abs().reshape(-1)
        code = torch.bucketize(a, mids)
        tie_up = (code < 7) & (a == mids[code.clamp(max=6)]) & ((code & 1) == 1)
        code = code + tie_up.to(code.dtype)
        neg = torch.signbit(y.reshape(-1)) & (code != 0)
        code = (code | (neg.to(code.dtype) << 3)).to(torch.uint8).view(-1, tokens)
        packed[r0:r0 + step] = code[:, 0::2] | (code[:, 1::2] << 4)
    byte = codes.astype(np.uint32).reshape(other, tokens // 64, 4)
    words = (byte[..., 0] | (byte[..., 1] << 8) | (byte[..., 2] << 16) | (byte[..., 3] << 24)).astype(np.uint32)
    return packed, torch.from_numpy(words.view(np.int32).T.copy())


def nvfp4_global_scale(x: torch.Tensor) -> float:
    """Per-tensor global scale (decode multiplier) that keeps every 16-token block scale within E4M3:
    amax / (6 * 448) as float32 (1 for an all-zero tensor)."""
    amax = float(x.abs().max())
    return float(np.float32(amax / (E2M1_MAX * E4M3_MAX))) if amax > 0 else 1.0


def pack_ragged_a(a2d: torch.Tensor, counts) -> torch.Tensor:
    """Re-store a logical [hidden, tokens_sum] A as per-expert K-contiguous blocks.

    Expert e's block is [hidden, n_e] row-major (leading dimension n_e) starting at
    element begin_e*hidden of the flat buffer ("tensor_ragged" input order).
    """
    hidden = a2d.shape[0]
    parts = []
    begin = 0
    for n in np.asarray(counts).tolist():
        if n:
            parts.append(a2d[:, begin:begin + n].contiguous().reshape(-1))
        begin += n
    if not parts:
        return a2d.new_empty((0,))
    flat = torch.cat(parts)
    assert flat.numel() == hidden * begin
    return flat


def store_operands(w: Workload, a_logical: torch.Tensor, b_logical: torch.Tensor):
    """Lay out logical A [hidden, tokens] and B [tokens, intermediate] as the workload stores them."""
    if w.a_major == "mn":
        a_store = a_logical.t().contiguous()
    elif w.input_order == "ragged":
        a_store = pack_ragged_a(a_logical, w.counts)
    else:
        a_store = a_logical
    if w.b_major == "k":
        bt = b_logical.t().contiguous()
        b_store = pack_ragged_a(bt, w.counts) if w.input_order == "ragged" else bt
    else:
        b_store = b_logical
    return a_store, b_store


def make_inputs(w: Workload, device="cpu") -> Inputs:
    """Draw the inputs of workload ``w`` on the CPU (seeded) and move them to ``device``."""
    gen = torch.Generator().manual_seed(int(w.seed))
    H, I, T, E = w.hidden, w.intermediate, w.tokens_sum, w.num_experts
    a32 = _normal(gen, (H, T), w.a_std)
    b32 = _normal(gen, (T, I), w.b_std)
    sfa = sfb = None
    if w.fp4:
        assert w.a_major == "k" and w.b_major == "k"
        gsa = gsb = None
        if w.sf_format == "ue4m3_16":
            # NVFP4: 16-token blocks on the pages' 256-token counts (blocks never cross experts)
            assert np.all(np.asarray(w.counts) % 64 == 0)
            ga, gb = nvfp4_global_scale(a32), nvfp4_global_scale(b32)
            a_store, sfa = quantize_e2m1_ue4m3_16(a32, 1, ga)
            b_store, sfb = quantize_e2m1_ue4m3_16(b32, 0, gb)
            gsa, gsb = torch.tensor([ga], dtype=torch.float32), torch.tensor([gb], dtype=torch.float32)
        else:
            a_store, sfa = quantize_per_expert(quantize_e2m1_ue8m0_32, a32, 1, w.counts, packed_fp4=True)  # [H, T/2]
            b_store, sfb = quantize_per_expert(quantize_e2m1_ue8m0_32, b32, 0, w.counts, packed_fp4=True)  # [I, T/2]
        if w.input_order == "ragged":   # per-expert [rows, n_e/2]-byte blocks back to back
            half = np.asarray(w.counts) // 2
            a_store, b_store = pack_ragged_a(a_store, half), pack_ragged_a(b_store, half)
        del a32, b32
        c = _normal(gen, (E, H, I), w.c_std).to(out_torch_dtype(w.out_dtype)) if w.accumulate else None
        offsets = torch.from_numpy(w.offsets.astype(np.int32))
        to = lambda t: None if t is None else t.to(device)
        return Inputs(to(a_store), to(b_store), to(offsets), to(sfa), to(sfb), to(c), to(gsa), to(gsb))
    if w.fp8 and w.sf_format == "ue8m0_32":
        a_store, sfa = quantize_per_expert(quantize_e4m3_ue8m0_32, a32, 1, w.counts)
        b_store, sfb = quantize_per_expert(quantize_e4m3_ue8m0_32, b32, 0, w.counts)
    elif w.fp8 and w.sf_format == "f32_any":
        a_store, sfa = quantize_per_expert(quantize_e4m3_fp32_blocks, a32, 1, w.counts)
        b_store, sfb = quantize_per_expert(quantize_e4m3_fp32_blocks, b32, 0, w.counts)
    elif w.fp8:
        a_store, sfa = quantize_per_expert(quantize_e4m3_blocks, a32, 1, w.counts)
        b_store, sfb = quantize_per_expert(quantize_e4m3_blocks, b32, 0, w.counts)
    else:
        a_store = a32.to(torch.bfloat16)
        b_store = b32.to(torch.bfloat16)
    del a32, b32
    a_store, b_store = store_operands(w, a_store, b_store)
    c = None
    if w.accumulate:
        c = _normal(gen, (E, H, I), w.c_std).to(out_torch_dtype(w.out_dtype))
    offsets = torch.from_numpy(w.offsets.astype(np.int32))
    to = lambda t: None if t is None else t.to(device)
    return Inputs(to(a_store), to(b_store), to(offsets), to(sfa), to(sfb), to(c))


def make_inputs_device(w: Workload, device) -> Inputs:
    """Same recipe as ``make_inputs`` but drawn with a device generator (fast, for timing only).

    The values differ from ``make_inputs``; shapes, dtypes and distributions are identical.
    """
    gen = torch.Generator(device=device).manual_seed(int(w.seed))
    H, I, T, E = w.hidden, w.intermediate, w.tokens_sum, w.num_experts

    def normal(shape, std, dtype):
        x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(dtype)

    if w.fp8 or w.fp4:
        cpu = make_inputs(w, "cpu")   # quantisation recipe lives on the CPU side
        to = lambda t: None if t is None else t.to(device)
        return Inputs(to(cpu.a), to(cpu.b), to(cpu.offsets), to(cpu.sfa), to(cpu.sfb), to(cpu.c), to(cpu.gsa),
                      to(cpu.gsb))
    a = normal((H, T), w.a_std, torch.bfloat16)
    b = normal((T, I), w.b_std, torch.bfloat16)
    a, b = store_operands(w, a, b)
    c = normal((E, H, I), w.c_std, out_torch_dtype(w.out_dtype)) if w.accumulate else None
    offsets = torch.from_numpy(w.offsets.astype(np.int32)).to(device)
    return Inputs(a, b, offsets, None, None, c)
