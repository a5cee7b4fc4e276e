"""Pins of the indexer oracle (oracle/index.py) to things other than itself:
the page's 9-token example (a query's candidates are its ancestor chain), the
ReLU clipping, closed-form orderings, the tie rule, and brute force against
the visible-key predicate."""
import numpy as np
import pytest

from conftest import golden
from oracle import attn as OA
from oracle import index as OI
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W


def _mask9_plan():
    g = golden("mask9.json")
    seqs = [np.asarray(s, np.int32) for s in g["seqs"]]
    tr = [np.zeros(len(s), np.uint8) for s in seqs]
    return g, OP.pack(seqs, tr, g["row_len"], g["min_shared"])


def test_mask9_query7_picks_only_its_ancestor_chain():
    """[P1] attention section: query 7 (branch B) sees R and B up to itself;
    with k at least the number of candidates, its top-k is exactly that set,
    and never branch A, whatever the scores of A's keys."""
    g, plan = _mask9_plan()
    T, H, D = 9, 2, 4
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, T, H, D))
    k = rng.standard_normal((1, T, D))
    k[0, 3:6] = 100.0 * np.abs(q[0, 7, 0])           # branch A would win every score
    w = np.ones((1, T, H))
    idx, _ = OI.topk(plan, q, k, w, top_k=8)
    assert list(idx[0, 7][idx[0, 7] >= 0]) == g["visible_of_query_7"]
    idx3, _ = OI.topk(plan, q, k, w, top_k=3)
    assert set(idx3[0, 7]) <= set(g["visible_of_query_7"])


def test_closed_form_ordering_and_ties():
    """k_j = j e_1, q_i = e_1, one head, w = 1: score(i, j) = j, so the top-k
    of a causal chain is its k largest visible indices; with all scores equal
    the tie rule keeps the k smallest indices."""
    T = 40
    seqs = [np.arange(T, dtype=np.int32) + 5]
    plan = OP.pack(seqs, [np.zeros(T, np.uint8)], 64, 64)
    q = np.zeros((1, 64, 1, 3))
    q[..., 0] = 1.0
    k = np.zeros((1, 64, 3))
    k[0, :, 0] = np.arange(64)
    w = np.ones((1, 64, 1))
    idx, val = OI.topk(plan, q, k, w, top_k=5)
    for i in range(T):
        want = list(range(max(0, i - 4), i + 1))
        assert list(idx[0, i][idx[0, i] >= 0]) == want
        np.testing.assert_allclose(val[0, i][: len(want)], want)
    k[0, :, 0] = 1.0                                    # all scores 1
    idx, _ = OI.topk(plan, q, k, w, top_k=5)
    for i in range(T):
        assert list(idx[0, i][idx[0, i] >= 0]) == list(range(min(5, i + 1)))


def test_relu_clips_negative_heads():
    """A head whose dot product is negative contributes 0, not a negative score."""
    T = 4
    plan = OP.pack([np.arange(T, dtype=np.int32)], [np.zeros(T, np.uint8)], 8, 64)
    q = np.zeros((1, 8, 2, 1))
    q[0, :, 0, 0] = 1.0
    q[0, :, 1, 0] = -1.0
    k = np.ones((1, 8, 1)) * 2.0
    w = np.ones((1, 8, 2)) * 3.0
    _, val = OI.topk(plan, q, k, w, top_k=2)
    assert np.allclose(val[0, 3, :2], 6.0)              # 3 * relu(2) + 3 * relu(-2)


@pytest.mark.parametrize("seed", range(3))
def test_brute_force_against_predicate(seed):
    """Random trees: the selection equals a brute-force top-k over the keys the
    predicate matrix marks visible (scores recomputed with einsum)."""
    b = W.random_forest(seed, n_roots=2, max_depth=3, max_children=3, len_lo=4, len_hi=30, row_len=256,
                        min_shared=8, vocab=W.VOCAB)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(seed)
    R, T, H, D, kk = plan.n_rows, plan.row_len, 3, 8, 7
    q = rng.standard_normal((R, T, H, D))
    k = rng.standard_normal((R, T, D))
    w = rng.random((R, T, H))
    idx, val = OI.topk(plan, q, k, w, top_k=kk)
    for r in range(R):
        M = OA.RowTree(plan, r).predicate_matrix()
        S = np.einsum("ihd,jd->ijh", q[r], k[r])
        S = np.einsum("ijh,ih->ij", np.maximum(S, 0), w[r])
        for i in range(T):
            cand = np.flatnonzero(M[i])
            best = cand[np.lexsort((cand, -S[i, cand]))][:kk]
            assert list(idx[r, i][idx[r, i] >= 0]) == sorted(best)
            np.testing.assert_allclose(val[r, i][: len(best)], S[i, sorted(best)], rtol=1e-12, atol=1e-12)
