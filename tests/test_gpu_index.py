"""Tree-aware top-k indexer on the GPU (stp_index_topk) against the oracle.

Exact: every selected key is a visible key of the query (its ancestor chain),
the count is min(k, candidates), keys are ascending and padded with -1.
Scores (bf16 products summed in float32 on the tensor cores) match the
float64 oracle on the same bf16 inputs within 1e-3 (1 + max |score|); the
selection is checked with that margin around the oracle's k-th score: every
key clearly above it is selected, none clearly below it is.
"""
import numpy as np
import pytest
import torch

from conftest import golden
from gpu_helpers import pack_both
from oracle import attn as OA
from oracle import index as OI
from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(se: np.ndarray, q, k, w, top_k, pairs=None):
    R, T = se.shape
    H, D = q.shape[2], q.shape[3]
    if pairs is None:
        pairs = stp.stp_count_tile_pairs(se)
    adesc = stp.Desc(R, T, 1, 1, 128, stp.STP_BF16, 0.1, pairs)
    buf = stp.Buffers(adesc)
    se_d = torch.from_numpy(np.ascontiguousarray(se)).cuda()
    stp.stp_classify(adesc, se_d, buf.tile_meta)
    idesc = stp.index_desc(R, T, H, D, top_k, pairs)
    ws = torch.empty(stp.stp_index_workspace_size(idesc), dtype=torch.uint8, device="cuda")
    idx = torch.empty(R, T, top_k, dtype=torch.int32, device="cuda")
    sc = torch.empty(R, T, top_k, dtype=torch.float32, device="cuda")
    stp.stp_index_topk(idesc, q.cuda(), k.cuda(), w.cuda(), se_d, buf.tile_meta, idx, sc, ws)
    torch.cuda.synchronize()
    assert stp.stp_device_status(buf.tile_meta) == stp.STP_OK
    status = stp.stp_device_status(ws)
    return idx.cpu().numpy(), sc.cpu().numpy(), status


def _check_query(rt, i, qn, kn, wn, top_k, gi, gs):
    cand = rt.visible(i)
    s = OI.scores(qn, kn, wn, i, cand)
    n = min(top_k, len(cand))
    sel = gi[gi >= 0]
    assert len(sel) == n and np.all(gi[n:] == -1) and np.all(np.isneginf(gs[n:]))
    assert np.all(np.diff(sel) > 0)
    pos = np.searchsorted(cand, sel)
    assert np.all(pos < len(cand)) and np.array_equal(cand[pos], sel), "a non-ancestor key was selected"
    tol = 1e-3 * (1.0 + np.abs(s).max())
    np.testing.assert_allclose(gs[:n], s[pos], atol=tol, rtol=0)
    if len(cand) > top_k:
        thr = np.sort(s)[::-1][top_k - 1]
        chosen = np.zeros(len(cand), bool)
        chosen[pos] = True
        assert np.all(chosen[s > thr + tol]), "a clearly better key was left out"
        assert np.all(s[chosen] >= thr - tol), "a clearly worse key was selected"


def test_mask9_query7_ancestor_chain_only(stp_lib):
    """[P1] attention section example: query 7 (branch B) gets exactly R and B
    up to itself, although branch A's keys would score highest."""
    g = golden("mask9.json")
    seqs = [np.asarray(s, np.int32) for s in g["seqs"]]
    tr = [np.zeros(len(s), np.uint8) for s in seqs]
    b = W.SeqBatch(seqs, tr, None, 128, g["min_shared"])
    out, info, ref = pack_both(b)
    q, k, w = W.index_tensors(1, 128, 2, 64, seed=3)
    k = k.float()
    k[0, 3:6] = 20.0 * q[0, 7].float().abs().sum(0) / 64      # branch A aligned with query 7
    k = k.to(torch.bfloat16)
    idx, sc, st = _run(out["subtree_end"], q, k, w, top_k=8)
    assert st == stp.STP_OK
    assert list(idx[0, 7][idx[0, 7] >= 0]) == g["visible_of_query_7"]


@pytest.mark.parametrize("top_k", [1, 7, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_random_forest_every_query(stp_lib, seed, top_k):
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=8, len_hi=160, row_len=1024,
                        min_shared=16, vocab=W.VOCAB)
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    R, T = se.shape
    q, k, w = W.index_tensors(R, T, 4, 64, seed=seed)
    idx, sc, st = _run(se, q, k, w, top_k)
    assert st == stp.STP_OK
    qn, kn, wn = q.double().numpy(), k.double().numpy(), w.double().numpy()
    for r in range(R):
        rt = OA.RowTree(ref, r)
        for i in range(T):
            _check_query(rt, i, qn[r], kn[r], wn[r], top_k, idx[r, i], sc[r, i])


@pytest.mark.parametrize("heads,dim", [(8, 64), (4, 128)])
def test_grpo_sampled_queries(stp_lib, heads, dim):
    """The 16384-token GRPO row (5000-token prefix + 16 rollouts), k = 512."""
    b = W.CONFIG_BATCHES["grpo"](W.CONFIG_SEEDS["grpo"])
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    q, k, w = W.index_tensors(1, b.row_len, heads, dim, seed=5)
    idx, sc, st = _run(se, q, k, w, top_k=512)
    assert st == stp.STP_OK
    qn, kn, wn = q.double().numpy()[0], k.double().numpy()[0], w.double().numpy()[0]
    rt = OA.RowTree(ref, 0)
    rng = np.random.default_rng(0)
    for i in list(rng.integers(0, b.row_len, size=24)) + [0, 300, 4999, 5000, b.row_len - 1]:
        _check_query(rt, int(i), qn, kn, wn, 512, idx[0, i], sc[0, i])


@pytest.mark.parametrize("top_k", [5, 100, 512])
def test_exact_ties_go_to_smaller_keys(stp_lib, top_k):
    """Scores with exact ties: every key row is one of three vectors (so a
    query's scores take at most three values, each computed identically),
    and with w = 0 every score is 0.  The selection is then unique: by score,
    ties to the smaller key index; compared exactly, on random forests and
    the GRPO row's first, middle and last query tiles."""
    cases = []
    b = W.random_forest(5, n_roots=3, max_depth=3, max_children=3, len_lo=8, len_hi=300, row_len=2048,
                        min_shared=16, vocab=W.VOCAB)
    cases.append(b)
    cases.append(W.CONFIG_BATCHES["grpo"](W.CONFIG_SEEDS["grpo"]))
    for bi, b in enumerate(cases):
        out, info, ref = pack_both(b)
        se = out["subtree_end"]
        R, T = se.shape
        q, k, w = W.index_tensors(R, T, 2, 64, seed=11 + bi)
        g = torch.Generator().manual_seed(7 + bi)
        basis = torch.randn(3, 64, generator=g) * torch.tensor([[1.0], [2.0], [4.0]])
        pick = torch.randint(0, 3, (R, T), generator=g)
        k = basis[pick].to(torch.bfloat16)
        for zero_w in (False, True):
            wc = torch.zeros_like(w) if zero_w else w
            idx, sc, st = _run(se, q, k, wc, top_k)
            assert st == stp.STP_OK
            qn, kn, wn = q.double().numpy(), k.double().numpy(), wc.double().numpy()
            queries = range(T) if T <= 2048 else [*range(0, 128), *range(8192, 8320), *range(T - 128, T)]
            for r in range(R):
                rt = OA.RowTree(ref, r)
                for i in queries:
                    cand = rt.visible(i)
                    s = OI.scores(qn[r], kn[r], wn[r], i, cand)
                    order = np.lexsort((cand, -s))[:top_k]
                    want = np.sort(cand[order])
                    got = idx[r, i][idx[r, i] >= 0]
                    assert np.array_equal(got, want), (bi, zero_w, r, i)
                    if zero_w:
                        assert np.all(sc[r, i][: len(want)] == 0.0)


def test_capacity_too_small_is_flagged(stp_lib):
    b = W.random_forest(3, n_roots=2, max_depth=2, max_children=3, len_lo=8, len_hi=100, row_len=512,
                        min_shared=16, vocab=W.VOCAB)
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    need = stp.stp_count_tile_pairs(se)
    R, T = se.shape
    q, k, w = W.index_tensors(R, T, 2, 64, seed=1)
    adesc = stp.Desc(R, T, 1, 1, 128, stp.STP_BF16, 0.1, need)
    buf = stp.Buffers(adesc)
    se_d = torch.from_numpy(se).cuda()
    stp.stp_classify(adesc, se_d, buf.tile_meta)
    idesc = stp.index_desc(R, T, 2, 64, 4, need - 1)
    ws = torch.empty(stp.stp_index_workspace_size(idesc), dtype=torch.uint8, device="cuda")
    idx = torch.empty(R, T, 4, dtype=torch.int32, device="cuda")
    sc = torch.empty(R, T, 4, dtype=torch.float32, device="cuda")
    stp.stp_index_topk(idesc, q.cuda(), k.cuda(), w.cuda(), se_d, buf.tile_meta, idx, sc, ws)
    torch.cuda.synchronize()
    assert stp.stp_device_status(ws) == stp.STP_EDEVICE


def test_descriptor_checks(stp_lib):
    for bad in (stp.index_desc(1, 256, 8, 96, 4), stp.index_desc(1, 256, 16, 64, 4),
                stp.index_desc(1, 256, 2, 64, 0), stp.index_desc(1, 200, 2, 64, 4)):
        with pytest.raises(stp.StpError):
            stp.stp_index_workspace_size(bad)
