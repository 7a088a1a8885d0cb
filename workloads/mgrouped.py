"""Seeded synthetic inputs for the M-grouped MoE GEMM (forward / dgrad of a grouped linear).

Draws inputs only: none of the method's arithmetic lives here, so the CUDA path and the
CPU oracle consume the same tensors without sharing any computation.

Shapes follow "05 · Grouped GEMM 与 Expert 计算", sections 2 and 5: A holds the tokens of all
groups ([M_total, K] contiguous, or [G, max_m, K] masked), B the per-group weights ([G, N, K]
K-major for the forward, [G, K, N] N-major for the dgrad), and D the output rows. Per-group
row counts use the uniform(0.7, 1.3) spread around an expected count that section 2.1 gives for
DeepGEMM's m-grouped generator, rounded to the nearest multiple of 128 for the contiguous
layouts (the tile alignment of section 2.1); masked counts are unaligned integers capped at
max_m (section 2.2).

The named shapes are the forward and dgrad of the same MoE layer whose weight gradient the
balanced K-grouped workload computes (in_dim 2048, out_dim 4096, 8 experts of ~4096 tokens).

Randomness: counts (and, for the index layout, the order of the 128-row blocks) come from
``numpy.random.default_rng(seed)`` in that order; tensors from a CPU ``torch.Generator``
seeded with ``seed`` (draw order: A, B, then D's previous contents).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

MG_ALIGN = 128


def round_to_128(x) -> np.ndarray:
    """Nearest multiple of 128: 128 * floor(x / 128 + 0.5)."""
    return (MG_ALIGN * np.floor(np.asarray(x, dtype=np.float64) / MG_ALIGN + 0.5)).astype(np.int64)


@dataclasses.dataclass
class MGWorkload:
    name: str
    num_groups: int
    n: int
    k: int
    layout: str                 # "offsets" | "indices" | "masked"
    counts: np.ndarray          # rows per group (masked: valid rows per group)
    seed: int
    max_m: int = 0              # masked only: rows reserved per group
    b_major: str = "k"          # "k": B [G, N, K] (forward); "mn": B [G, K, N] (dgrad)
    out_dtype: str = "bf16"     # "f32" | "bf16" | "f16"
    accumulate: bool = False
    a_std: float = 1.0
    b_std: float = 0.02
    d_std: float = 1.0          # D's previous contents ~ N(0, d_std) (accumulate, masked)
    shuffle_blocks: bool = False  # index layout: 128-row blocks in random group order
    fp8: bool = False           # e4m3 operands, scales per row / column per 128 K (or UE8M0 per 32)
    sf_format: str = "f32_128"  # "f32_128" | "ue8m0_32"

    @property
    def m(self) -> int:
        """The ``m`` argument: rows of A (contiguous) or rows per group (masked)."""
        return self.max_m if self.layout == "masked" else int(np.asarray(self.counts).sum())

    @property
    def rows(self) -> int:
        return self.num_groups * self.max_m if self.layout == "masked" else self.m

    @property
    def valid_rows(self) -> int:
        return int(np.asarray(self.counts).sum())

    @property
    def flops(self) -> int:
        return 2 * self.valid_rows * self.n * self.k


def counts_spread(seed: int, num_groups: int, expected_m: int, aligned: bool, cap: Optional[int] = None):
    rng = np.random.default_rng(seed)
    x = expected_m * rng.uniform(0.7, 1.3, size=num_groups)
    c = round_to_128(x) if aligned else np.floor(x + 0.5).astype(np.int64)
    if cap is not None:
        c = np.minimum(c, cap)
    return c, rng


def mg_tiny() -> MGWorkload:
    return MGWorkload("M-grouped tiny: G=4 N=256 K=128 counts [128,256,0,384]", 4, 256, 128, "offsets",
                      np.array([128, 256, 0, 384]), seed=10)


def mg_forward() -> MGWorkload:
    c, _ = counts_spread(5, 8, 4096, aligned=True)
    return MGWorkload("M-grouped forward: G=8 rows ~4096 each, N=4096 K=2048, B [G,N,K], BF16 out",
                      8, 4096, 2048, "offsets", c, seed=5)


def mg_dgrad() -> MGWorkload:
    c, _ = counts_spread(6, 8, 4096, aligned=True)
    return MGWorkload("M-grouped dgrad: G=8 rows ~4096 each, N=2048 K=4096, B [G,K,N], BF16 out",
                      8, 2048, 4096, "offsets", c, seed=6, b_major="mn")


def mg_masked() -> MGWorkload:
    c, _ = counts_spread(7, 16, 256, aligned=False, cap=1024)
    return MGWorkload("M-grouped masked decode: G=16 max_m=1024 masked_m ~256, N=4096 K=2048, BF16 out",
                      16, 4096, 2048, "masked", c, seed=7, max_m=1024)


def mg_fp8_forward() -> MGWorkload:
    c, _ = counts_spread(5, 8, 4096, aligned=True)
    return MGWorkload("M-grouped FP8 forward: G=8 rows ~4096 each, N=4096 K=2048, e4m3 with per-128-K FP32 scales, "
                      "BF16 out", 8, 4096, 2048, "offsets", c, seed=11, fp8=True, b_std=1.0)


def mg_fp8_masked() -> MGWorkload:
    c, _ = counts_spread(7, 16, 256, aligned=False, cap=1024)
    return MGWorkload("M-grouped FP8 masked decode: G=16 max_m=1024 masked_m ~256, N=4096 K=2048, e4m3, BF16 out",
                      16, 4096, 2048, "masked", c, seed=12, max_m=1024, fp8=True, b_std=1.0)


MG_NAMED = {"mg_tiny": mg_tiny, "mg_forward": mg_forward, "mg_dgrad": mg_dgrad, "mg_masked": mg_masked,
            "mg_fp8_forward": mg_fp8_forward, "mg_fp8_masked": mg_fp8_masked}


def mg_custom(num_groups: int, n: int, k: int, layout: str, counts, seed: int, **kw) -> MGWorkload:
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.shape == (num_groups,)
    return MGWorkload(f"custom M-grouped G={num_groups} N={n} K={k} {layout}", num_groups, n, k, layout,
                      counts, seed, **kw)


@dataclasses.dataclass
class MGInputs:
    """a: bf16 [rows, K] (masked: [G, max_m, K]); b: bf16 [G, N, K] or [G, K, N];
    groups: int32 offsets [G] / m_indices [rows] / masked_m [G]; d0: D's previous contents
    ([rows, N] or [G, max_m, N]) in the output dtype, or None (overwrite of a contiguous layout,
    where every row is written). FP8: a, b are float8_e4m3fn of the same shapes; sfa float32
    [K/128, rows] (or packed UE8M0 int32 words of that shape), sfb [G, K/128, N]."""
    a: torch.Tensor
    b: torch.Tensor
    groups: torch.Tensor
    d0: Optional[torch.Tensor]
    sfa: Optional[torch.Tensor] = None
    sfb: Optional[torch.Tensor] = None


def group_ids(w: MGWorkload) -> np.ndarray:
    """Index layout: the group id of every row, blocks of 128 rows (optionally shuffled)."""
    blocks = np.repeat(np.arange(w.num_groups), np.asarray(w.counts) // MG_ALIGN)
    if w.shuffle_blocks:
        rng = np.random.default_rng(w.seed + 1000)
        blocks = blocks[rng.permutation(len(blocks))]
    return np.repeat(blocks, MG_ALIGN).astype(np.int32)


def groups_array(w: MGWorkload) -> np.ndarray:
    if w.layout == "offsets":
        return np.cumsum(np.asarray(w.counts, dtype=np.int64)).astype(np.int32)
    if w.layout == "indices":
        return group_ids(w)
    return np.asarray(w.counts, dtype=np.int32)


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[name]


def make_mg_inputs(w: MGWorkload, device="cpu", on_device_rng: bool = False) -> MGInputs:
    """Draw the inputs of ``w`` (seeded). ``on_device_rng`` draws with a device generator instead
    (same shapes and distributions, different values; for timing only)."""
    dev_gen = on_device_rng and str(device) != "cpu"
    gen = torch.Generator(device=device if dev_gen else "cpu").manual_seed(int(w.seed))

    def normal(shape, std, dtype):
        x = torch.randn(*shape, generator=gen, device=device if dev_gen else "cpu", dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(dtype)

    a_shape = (w.num_groups, w.max_m, w.k) if w.layout == "masked" else (w.rows, w.k)
    b_shape = (w.num_groups, w.n, w.k) if w.b_major == "k" else (w.num_groups, w.k, w.n)
    d_shape = (w.num_groups, w.max_m, w.n) if w.layout == "masked" else (w.rows, w.n)
    sfa = sfb = None
    if w.fp8:
        from . import quantize_e4m3_blocks, quantize_e4m3_ue8m0_32
        quant = quantize_e4m3_ue8m0_32 if w.sf_format == "ue8m0_32" else quantize_e4m3_blocks
        a32 = normal(a_shape, w.a_std, torch.float32).cpu()
        b32 = normal(b_shape, w.b_std, torch.float32).cpu()
        a, sfa = quant(a32.reshape(-1, w.k), token_axis=1)            # per row, per block of K
        a = a.reshape(a_shape)
        qb, sb = [], []
        for g in range(w.num_groups):                                 # per column, per block of K
            q, sc = quant(b32[g], token_axis=1 if w.b_major == "k" else 0)
            qb.append(q)
            sb.append(sc)
        b, sfb = torch.stack(qb), torch.stack(sb)
    else:
        a = normal(a_shape, w.a_std, torch.bfloat16)
        b = normal(b_shape, w.b_std, torch.bfloat16)
    d0 = normal(d_shape, w.d_std, _torch_dtype(w.out_dtype)) if (w.accumulate or w.layout == "masked") else None
    groups = torch.from_numpy(groups_array(w))
    to = lambda t: None if t is None else t.to(device)
    return MGInputs(to(a), to(b), to(groups), to(d0), to(sfa), to(sfb))
