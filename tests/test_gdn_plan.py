"""Host planner of the tree-aware Gated DeltaNet (stp_gdn_plan) against the
oracle's paths: the path predecessor of every token equals the one read off
the packer's parent pointers; segments are consecutive runs that break at
every branch point and start from their parent's last token (and a root run
of at least 32 chunks is cut once, after its first 16, into two segments);
depths are ordered; chunks of at most 64 tokens tile every segment exactly
once, on the same boundaries as without the cut."""
import numpy as np
import pytest

from oracle import gdn as OG
from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W


def _check(plan_o, H=2):
    R, T = plan_o.n_rows, plan_o.row_len
    desc = stp.gdn_desc(R, T, H)
    used = np.asarray(plan_o.used, np.int32)
    plan = stp.stp_gdn_plan(desc, plan_o.subtree_end, used)
    a = stp.gdn_plan_arrays(plan)
    prev = a["prev"]
    for r in range(R):
        want = OG.path_prev(plan_o, r)
        got = prev[r * T: (r + 1) * T].astype(np.int64)
        u = used[r]
        assert np.all(got[u:] == -2)
        exp = np.where(want[:u] >= 0, want[:u] + r * T, -1)
        assert np.array_equal(got[:u], exp)
    back = lambda a: np.where(a >= 0, prev[np.maximum(a, 0)], -1)  # noqa: E731
    p2 = back(prev)
    assert np.array_equal(a["prev2"], p2) and np.array_equal(a["prev3"], back(p2))
    n_child = np.bincount(prev[prev >= 0], minlength=R * T)
    covered = np.zeros(R * T, np.int64)
    depth = np.full(len(a["seg_start"]), -1)
    d_of = np.zeros(len(a["seg_start"]), np.int64)
    for d in range(len(a["depth_off"]) - 1):
        d_of[a["depth_off"][d]: a["depth_off"][d + 1]] = d
    for i, (s, L, par) in enumerate(zip(a["seg_start"], a["seg_len"], a["seg_parent"])):
        covered[s: s + L] += 1
        if par >= 0:
            ps, pl = a["seg_start"][par], a["seg_len"][par]
            assert prev[s] == ps + pl - 1, "a segment must start from its parent's last token"
            assert d_of[par] == d_of[i] - 1
            if prev[s] == s - 1 and n_child[s - 1] == 1 and s % T != 0:
                # no branch point here: the cut of a long root run after 16 chunks
                assert a["seg_parent"][par] < 0 and pl == 16 * 64 and L + pl >= 32 * 64
        else:
            assert prev[s] == -1 and d_of[i] == 0
        for x in range(s + 1, s + L):
            assert prev[x] == x - 1 and n_child[x - 1] == 1
        depth[i] = d_of[i]
        c0 = a["seg_chunk0"][i]
        n = (L + 63) // 64
        assert np.array_equal(a["chunk_start"][c0: c0 + n], s + 64 * np.arange(n))
        assert np.array_equal(a["chunk_len"][c0: c0 + n], np.minimum(64, L - 64 * np.arange(n)))
    kids = [[] for _ in a["seg_start"]]
    for i, par in enumerate(a["seg_parent"]):
        if par >= 0:
            kids[par].append(i)
    for i, want_kids in enumerate(kids):
        assert list(a["child"][a["child_off"][i]: a["child_off"][i + 1]]) == want_kids
    real = prev != -2
    assert np.all(covered[real] == 1) and np.all(covered[~real] == 0)
    # successor lists: exactly the tokens whose path predecessor is x, ascending
    so, sl = a["succ_off"], a["succ"]
    for x in np.flatnonzero(n_child > 0).tolist() + [0, R * T - 1]:
        assert list(sl[so[x]: so[x + 1]]) == list(np.flatnonzero(prev == x))
    assert so[-1] == int((prev >= 0).sum()) and np.array_equal(np.diff(so), np.bincount(prev[prev >= 0], minlength=R * T))
    assert a["seg_chunk0"][-1] + (a["seg_len"][-1] + 63) // 64 == len(a["chunk_start"])
    return plan


@pytest.mark.parametrize("seed", range(12))
def test_random_forests(seed):
    b = W.random_forest(seed, n_roots=3, max_depth=4, max_children=3, len_lo=1, len_hi=150, row_len=1024,
                        min_shared=4, vocab=41)
    _check(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared))


@pytest.mark.parametrize("name", ["tiny", "grpo", "deep", "bushy"])
def test_workloads(name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    _check(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared))


def test_no_row_used_means_every_token_is_real():
    b = W.tiny(0)
    p = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    plan = stp.stp_gdn_plan(stp.gdn_desc(1, p.row_len, 1), p.subtree_end)
    assert np.all(stp.gdn_plan_arrays(plan)["prev"] >= -1)


def test_rejections():
    desc = stp.gdn_desc(1, 8, 1)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_plan(desc, np.array([[9, 1, 2, 3, 4, 5, 6, 7]], np.int32))       # outside [x, T)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_plan(desc, np.array([[3, 1, 4, 3, 4, 5, 6, 7]], np.int32))       # not nested
    with pytest.raises(stp.StpError):
        stp.stp_gdn_plan(desc, np.arange(8, dtype=np.int32)[None], np.array([9], np.int32))
    plan = stp.stp_gdn_plan(desc, np.arange(8, dtype=np.int32)[None])
    with pytest.raises(stp.StpError):
        stp.stp_gdn_workspace_size(stp.gdn_desc(1, 8, 1, head_dim=64), plan)      # head_dim must be 128
    with pytest.raises(stp.StpError):
        stp.stp_gdn_workspace_size(stp.gdn_desc(1, 16, 1), plan)                  # plan of another size
    assert stp.stp_gdn_workspace_size(desc, plan) > 0
    with pytest.raises(stp.StpError):   # reaches the library (argument marshalling) and fails its checks
        stp.stp_gdn_fwd(stp.gdn_desc(1, 8, 1, head_dim=64), plan, None, None, None, None, None, None, None,
                        stream=0)


def test_edge_shapes():
    """No rows; rows of pads only; single-token rows; a row of one chain."""
    desc0 = stp.gdn_desc(0, 128, 2)
    plan0 = stp.stp_gdn_plan(desc0, np.zeros((0, 128), np.int32))
    assert plan0[stp.GP_N] == 0 and plan0[stp.GP_NSEG] == 0 and plan0[stp.GP_NCHUNK] == 0
    assert stp.stp_gdn_workspace_size(desc0, plan0) > 0
    T = 8
    se = np.tile(np.arange(T, dtype=np.int32), (3, 1))
    desc = stp.gdn_desc(3, T, 1)
    plan = stp.stp_gdn_plan(desc, se, np.array([0, 1, T], np.int32))   # all pads; one token; T isolated tokens
    a = stp.gdn_plan_arrays(plan)
    assert np.all(a["prev"][:T] == -2)
    assert a["prev"][T] == -1 and np.all(a["prev"][T + 1: 2 * T] == -2)
    assert np.all(a["prev"][2 * T:] == -1)          # subtree_end = own index: every token its own root
    assert len(a["seg_start"]) == 1 + T and np.all(a["seg_len"] == 1)
    chain = np.full((1, 200), 199, np.int32)         # one sequence: every token sees all before it
    plan = stp.stp_gdn_plan(stp.gdn_desc(1, 200, 1), chain)
    a = stp.gdn_plan_arrays(plan)
    assert np.array_equal(a["prev"], np.arange(200) - 1)
    assert list(a["seg_len"]) == [200] and list(a["chunk_len"]) == [64, 64, 64, 8]


@pytest.mark.parametrize("n", [2047, 2048, 3000])
def test_long_root_run_is_cut_once(n):
    """A root run of at least 32 chunks becomes two segments: its first 16
    chunks at depth 0, the rest their only child at depth 1; the chunks are
    the same as without the cut."""
    T = 4096
    chain = np.full((1, T), n - 1, np.int32)
    chain[0, n:] = np.arange(n, T)
    plan = stp.stp_gdn_plan(stp.gdn_desc(1, T, 1), chain, np.array([n], np.int32))
    a = stp.gdn_plan_arrays(plan)
    if n < 2048:
        assert list(a["seg_len"]) == [n] and list(a["seg_parent"]) == [-1]
        assert list(a["depth_off"]) == [0, 1]
    else:
        assert list(a["seg_start"]) == [0, 1024] and list(a["seg_len"]) == [1024, n - 1024]
        assert list(a["seg_parent"]) == [-1, 0] and list(a["depth_off"]) == [0, 1, 2]
        assert list(a["child"][a["child_off"][0]: a["child_off"][1]]) == [1]
    k = np.arange((n + 63) // 64)
    assert np.array_equal(a["chunk_start"], 64 * k) and np.array_equal(a["chunk_len"], np.minimum(64, n - 64 * k))
