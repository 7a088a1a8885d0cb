"""Expert placement across ranks for multi-GPU runs (host logic only, no arithmetic of the method).

Experts are independent units of the K-grouped weight-gradient GEMM: expert e's gradient
depends only on its own token range of A and B. Under expert parallelism each rank holds the
tokens of the experts placed on it and computes their gradients with no exchange step
("05 · Grouped GEMM 与 Expert 计算", introduction and section 2: experts distributed over
devices, each device running a grouped GEMM over its local experts). What a placement has to
do is keep the work per rank even; the work of expert e is proportional to its token count
n_e (2 * hidden * intermediate * n_e FLOPs), so ranks are balanced on the sum of n_e.

``assign_experts`` uses longest-processing-time-first list scheduling: experts in decreasing
token count (ties: lower index first) each go to the rank whose token sum is smallest so far
(ties: lower rank). Its per-rank sums differ by at most the largest single count. Each rank
keeps its experts in ascending index order, so a rank's local problem lists them as the global
problem does.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def assign_experts(counts: Sequence[int], world: int) -> List[List[int]]:
    """Per rank, the ascending list of experts it owns (every expert on exactly one rank)."""
    if world < 1:
        raise ValueError("world must be >= 1")
    c = [int(v) for v in np.asarray(counts).reshape(-1).tolist()]
    if any(v < 0 for v in c):
        raise ValueError("token counts must be non-negative")
    order = sorted(range(len(c)), key=lambda e: (-c[e], e))
    load = [0] * world
    owned: List[List[int]] = [[] for _ in range(world)]
    for e in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owned[r].append(e)
        load[r] += c[e]
    return [sorted(o) for o in owned]


def rank_token_sums(counts: Sequence[int], owned: Sequence[Sequence[int]]) -> List[int]:
    """Sum of n_e over each rank's experts."""
    c = np.asarray(counts, dtype=np.int64).reshape(-1)
    return [int(c[list(o)].sum()) if len(o) else 0 for o in owned]


def local_problem(counts: Sequence[int], experts: Sequence[int]) -> Tuple[np.ndarray, np.ndarray, List[Tuple[int, int]]]:
    """A rank's local problem: its experts' counts, their cumulative int32 offsets (the layout the
    library takes), and each expert's token range [begin_e, end_e) in the global problem, from
    which the rank's A columns and B rows are taken (in this order, back to back)."""
    c = np.asarray(counts, dtype=np.int64).reshape(-1)
    ends = np.cumsum(c)
    begins = ends - c
    local = c[list(experts)] if len(experts) else np.zeros(0, dtype=np.int64)
    offsets = np.cumsum(local).astype(np.int32)
    ranges = [(int(begins[e]), int(ends[e])) for e in experts]
    return local, offsets, ranges
