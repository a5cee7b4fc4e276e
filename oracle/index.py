"""Oracle: the tree-aware top-k indexer, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source (prefix-tree-packing page, attention section, the sparse top-k indexer
variants): top-k sparse attention gathers whatever key indices it is handed;
all tree awareness lives in the indexer, which only ever scores candidates
from a query's own ancestor chain -- the same enter/exit interval check as the
mask -- so keys of a sibling branch are never proposed, let alone selected.

The page names the indexer variants but prints no scoring formula; the
lightning-indexer form is taken (the plainest one for "score, then keep the
top k"): with H indexer heads, per-query head weights w and a key vector per
token,

    score(i, j) = sum_h w[i, h] * max(q[i, h] . k[j], 0)     for j in V(i)

where V(i) is query i's visible set (its ancestor segments and its own
segment up to i; a pad sees only itself).  The top-k of query i are the k
candidates of largest score, ties to the smaller key index; fewer than k
candidates are all kept.  The output lists the selected key indices in
ascending order (what a sparse attention kernel gathers), with their scores,
padded with index -1 and score -inf.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from .attn import RowTree
from .pack import Plan


def scores(q: np.ndarray, k: np.ndarray, w: np.ndarray, i: int, keys: np.ndarray) -> np.ndarray:
    """score(i, j) for the given keys j of one row; q [T, H, D], k [T, D], w [T, H]."""
    dots = np.asarray(k, np.float64)[keys] @ np.asarray(q, np.float64)[i].T   # [n_keys, H]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)[i]


def topk_query(rt: RowTree, i: int, q, k, w, top_k: int) -> Tuple[np.ndarray, np.ndarray]:
    """(selected key indices ascending, their scores) of query i of one row."""
    keys = rt.visible(i)
    s = scores(q, k, w, i, keys)
    order = np.lexsort((keys, -s))[:top_k]      # by score descending, then key ascending
    sel = np.sort(keys[order])
    return sel, scores(q, k, w, i, sel)


def topk(plan: Plan, q, k, w, top_k: int) -> Tuple[np.ndarray, np.ndarray]:
    """All queries of all rows: indices int32 [R, T, top_k], scores float64
    [R, T, top_k]; q [R, T, H, D], k [R, T, D], w [R, T, H]."""
    R, T = plan.n_rows, plan.row_len
    idx = np.full((R, T, top_k), -1, np.int32)
    val = np.full((R, T, top_k), -np.inf)
    for r in range(R):
        rt = RowTree(plan, r)
        for i in range(T):
            sel, sc = topk_query(rt, i, q[r], k[r], w[r], top_k)
            idx[r, i, :len(sel)] = sel
            val[r, i, :len(sel)] = sc
    return idx, val
