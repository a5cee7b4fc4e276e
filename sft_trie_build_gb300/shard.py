"""Splitting the attention path across ranks (one process per GPU).

Packed rows are independent, and within a row every kv-head group is
independent (dK/dV reduce only over the query heads of their own group), so
the path partitions into units (row, kv head) with no exchange step.  Two
ways of using several GPUs follow:

* weak scaling (bench.py): every rank packs and processes its own batch,
  drawn with its own seed;
* one batch split across ranks: ``shard_units_weighted`` assigns each rank
  a contiguous range of units holding about the same attention work (the
  useful (query, key) pairs of a row, the same for each of its kv heads;
  ``row_useful_pairs`` counts them), ``shard_units`` the same number of
  units, and ``unit_runs`` turns a range into (row, first kv head, end kv
  head) launches.

The only collective is ``max_over_ranks`` on timings, never on data.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of the batch a rank draws under weak scaling."""
    return base_seed + 1000 * rank


def shard_units(n_rows: int, n_kv_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """Half-open range [u0, u1) of units u = row * n_kv_heads + kv_head owned by
    `rank`; ranges are contiguous, disjoint, cover every unit and differ in
    size by at most one."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    n = n_rows * n_kv_heads
    base, extra = divmod(n, world)
    u0 = rank * base + min(rank, extra)
    return u0, u0 + base + (1 if rank < extra else 0)


def row_useful_pairs(position_ids, used) -> np.ndarray:
    """Useful (query, key) pairs of each packed row: a real token at position
    p sees p + 1 keys (its ancestors and itself), so a row's work is the sum
    of (p + 1) over its first used[r] tokens."""
    pos = np.asarray(position_ids, np.int64)
    used = np.asarray(used, np.int64)
    cols = np.arange(pos.shape[1])[None, :]
    return np.where(cols < used[:, None], pos + 1, 0).sum(1)


def shard_units_weighted(row_work, n_kv_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """Half-open range [u0, u1) of units u = row * n_kv_heads + kv_head owned
    by `rank`, unit u weighing row_work[u // n_kv_heads]: rank k's range
    starts at the first unit whose preceding work reaches k / world of the
    total.  Ranges are contiguous, disjoint and cover every unit; a rank's
    work exceeds total / world by less than one unit's weight."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    w = np.repeat(np.asarray(row_work, np.float64), n_kv_heads)
    before = np.concatenate([[0.0], np.cumsum(w)])[:-1]   # work of the units before u
    total = float(w.sum())

    def start(k):
        if k <= 0:
            return 0
        if k >= world:
            return len(w)
        return int(np.searchsorted(before, total * k / world, side="left"))

    return start(rank), start(rank + 1)


def unit_runs(u0: int, u1: int, n_kv_heads: int) -> List[Tuple[int, int, int]]:
    """Split a unit range into per-row launches (row, g0, g1): kv heads
    [g0, g1) of that row (query heads [g0 G, g1 G))."""
    out = []
    u = u0
    while u < u1:
        r, g0 = divmod(u, n_kv_heads)
        g1 = min(n_kv_heads, g0 + (u1 - u))
        out.append((r, g0, g1))
        u += g1 - g0
    return out


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a float over all ranks of the default process group (the
    value itself when torch.distributed is not initialized)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
