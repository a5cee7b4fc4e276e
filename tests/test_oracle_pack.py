"""Pins of the packing oracle against the pages and against mathematics."""
import itertools

import numpy as np
import pytest

from conftest import golden
from oracle import pack as P
from oracle.attn import RowTree
from sft_trie_build_gb300 import workloads as W


def _private_batch(sizes):
    seqs = [np.arange(1000 * (i + 1), 1000 * (i + 1) + n, dtype=np.int32) for i, n in enumerate(sizes)]
    tr = [np.ones(n, np.uint8) for n in sizes]
    return seqs, tr


# --- worked examples printed on the pages --------------------------------

def test_rollout32_global_and_in_order():
    g = golden("rollout32.json")
    b = W.rollout32(0)
    glob = P.pack(b.seqs, b.trainable, g["row_len"], 64, b.family)
    assert glob.used == g["global_used"]
    assert glob.n_rows * g["row_len"] == g["allocated_global"]
    ino = P.pack(b.seqs, b.trainable, g["row_len"], 64, b.family, in_order=True)
    assert ino.used == g["in_order_used"]
    assert ino.n_rows * g["row_len"] == g["allocated_in_order"]
    # row contents: long + 3 short A | medium + 5 short A + short B
    fam_rows = [sorted(int(b.family[lf.seq]) for lf in bn.leaves) for bn in glob.bins]
    assert fam_rows[0] == [0, 0, 0] + [2] * 8
    assert fam_rows[1] == [0] * 5 + [1] * 8 + [3] * 8


def test_rollout32_accounting():
    """11,999 shared group-prefix tokens, completion + 1 per rollout, root once."""
    b = W.rollout32(0)
    plan = P.pack(b.seqs, b.trainable, 131072, 64, b.family)
    lens = sorted(seg.length for seg in plan.trie.segments)
    assert lens.count(11999) == 4 and lens.count(4096) == 1
    comp = {0: 2000, 1: 2000, 2: 12000, 3: 7000}
    for s in range(32):
        leaf = plan.trie.segments[plan.trie.leaf_of[s]]
        assert leaf.length == comp[int(b.family[s])] + 1


def test_mask_example_nine_tokens():
    g = golden("mask9.json")
    seqs = [np.array(s, np.int32) for s in g["seqs"]]
    tr = [np.zeros(len(s), np.uint8) for s in seqs]
    plan = P.pack(seqs, tr, g["row_len"], g["min_shared"])
    assert plan.n_rows == 1
    assert plan.token_ids[0].tolist() == g["token_ids"]
    assert plan.subtree_end[0].tolist() == g["subtree_end"]
    rt = RowTree(plan, 0)
    assert rt.visible(7).tolist() == g["visible_of_query_7"]


@pytest.mark.parametrize("case", golden("bfd_small.json")["cases"], ids=lambda c: c["name"])
def test_bfd_hand_worked(case):
    seqs, tr = _private_batch(case["sizes"])
    fam = None if case["family"] is None else np.array(case["family"], np.int32)
    plan = P.pack(seqs, tr, case["row_len"], 64, fam)
    assert [sorted(lf.seq for lf in bn.leaves) for bn in plan.bins] == case["bins"]
    assert plan.used == case["used"]


# --- classical bin packing facts ------------------------------------------

def _opt_bins(sizes, cap):
    """Exact minimum number of bins by exhaustive search (tiny inputs)."""
    n = len(sizes)
    best = n
    for assign in itertools.product(range(n), repeat=n):
        if max(assign) + 1 >= best:
            continue
        loads = [0] * n
        ok = True
        for i, a in enumerate(assign):
            loads[a] += sizes[i]
            if loads[a] > cap:
                ok = False
                break
        if ok:
            best = max(assign) + 1
    return best


@pytest.mark.parametrize("seed", range(12))
def test_private_segments_are_classical_bin_packing(seed):
    rng = np.random.default_rng(seed)
    cap = 20
    sizes = [int(x) for x in rng.integers(1, cap + 1, size=int(rng.integers(3, 7)))]
    seqs, tr = _private_batch(sizes)
    plan = P.pack(seqs, tr, cap, 64)
    # loads are plain sums of item sizes
    for bn, u in zip(plan.bins, plan.used):
        assert u == sum(sizes[lf.seq] for lf in bn.leaves) <= cap
    opt = _opt_bins(sizes, cap)
    nb = plan.n_rows
    assert nb >= opt >= -(-sum(sizes) // cap)
    # best-fit-decreasing guarantee (Johnson 1973): BFD <= 11/9 OPT + 4
    assert nb <= 11 / 9 * opt + 4
    # any-fit property: at most one bin is at most half full
    assert sum(1 for u in plan.used if 2 * u <= cap) <= 1


# --- closed forms and structural invariants -------------------------------

def _prefix_free_batch(seed, n_prompts=5, per_prompt=3, vocab=6):
    """Prefix-free non-trainable prompts over a small vocabulary (so prompts
    share random stretches) followed by trainable completions."""
    rng = np.random.default_rng(seed)
    prompts = []
    while len(prompts) < n_prompts:
        p = tuple(int(x) for x in rng.integers(0, vocab, int(rng.integers(2, 9))))
        if any(p[:len(q)] == q or q[:len(p)] == p for q in prompts):
            continue
        prompts.append(p)
    seqs, tr = [], []
    for p in prompts:
        for _ in range(int(rng.integers(1, per_prompt + 1))):
            c = rng.integers(0, vocab, int(rng.integers(1, 6)))
            seqs.append(np.array(list(p) + list(c), np.int32))
            tr.append(np.array([0] * len(p) + [1] * len(c), np.uint8))
    return seqs, tr


def _closed_form_tokens(seqs, tr):
    """|{distinct s[:k], 1 <= k <= c(s)}| + sum (len(s) - c(s)), where
    c(s) = nt(s) - [nt(s) < len(s)]: non-trainable prefixes are shared up to
    the copied context token, everything after it is private."""
    return _distinct_prefixes(seqs, tr, True) + sum(
        len(s) - _cap(s, t) for s, t in zip(seqs, tr))


def _cap(s, t):
    nt = P.leading_nontrainable(t)
    return max(0, nt - (1 if nt < len(s) else 0))


def _distinct_prefixes(seqs, tr=None, capped=False):
    """Number of distinct non-empty prefixes (a character trie's node count),
    counted by inserting every sequence into nested dicts."""
    root, nodes = {}, 0
    for i, s in enumerate(seqs):
        n = _cap(s, tr[i]) if capped else len(s)
        cur = root
        for x in s[:n].tolist():
            nxt = cur.get(x)
            if nxt is None:
                nxt = cur[x] = {}
                nodes += 1
            cur = nxt
    return nodes


@pytest.mark.parametrize("seed", range(20))
def test_trie_token_count_closed_form(seed):
    seqs, tr = _prefix_free_batch(seed)
    plan = P.pack(seqs, tr, 100000, min_shared=1)
    assert plan.n_rows == 1
    assert plan.used[0] == _closed_form_tokens(seqs, tr)
    # a larger minimum can only add tokens
    plan64 = P.pack(seqs, tr, 100000, min_shared=64)
    assert plan64.used[0] >= plan.used[0]


@pytest.mark.parametrize("seed", range(10))
def test_all_nontrainable_is_plain_trie(seed):
    """No trainable tokens, min 1: the row holds one token per distinct
    non-empty prefix (textbook trie node count)."""
    rng = np.random.default_rng(100 + seed)
    seqs = [rng.integers(0, 3, int(rng.integers(1, 8))).astype(np.int32) for _ in range(8)]
    tr = [np.zeros(len(s), np.uint8) for s in seqs]
    plan = P.pack(seqs, tr, 100000, min_shared=1)
    distinct = {tuple(int(x) for x in s[:k]) for s in seqs for k in range(1, len(s) + 1)}
    assert plan.used[0] == len(distinct) == _distinct_prefixes(seqs)


@pytest.mark.parametrize("name", ["grpo", "deep"])
def test_min64_equals_closed_form_when_runs_are_long(name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    plan = P.pack(b.seqs, b.trainable, b.row_len, 64, b.family)
    assert plan.used[0] == _closed_form_tokens(b.seqs, b.trainable)


def _check_layout(plan, seqs, tr, min_shared):
    T = plan.row_len
    offs = np.concatenate([[0], np.cumsum([len(s) for s in seqs])])
    flat_tok = plan.token_ids.reshape(-1)
    flat_pos = plan.position_ids.reshape(-1)
    flat_lm = plan.loss_mask.reshape(-1)
    users = {}
    for s, (seq, t) in enumerate(zip(seqs, tr)):
        g = plan.gather_index[offs[s]:offs[s + 1]]
        rows = set((g // T).tolist())
        assert len(rows) == 1                       # one leaf, one row
        assert (flat_tok[g] == seq).all()           # sequence reconstructs
        assert (flat_pos[g] == np.arange(len(seq))).all()
        assert (np.diff(g) > 0).all()               # DFS order keeps positions increasing
        nxt = np.concatenate([t[1:], [0]]).astype(np.uint8)
        assert (flat_lm[g] == nxt).all()
        for p, x in enumerate(g.tolist()):
            users.setdefault(x, []).append((s, p))
        # loss positions are followed in the row by the token they predict
        lp = np.flatnonzero(nxt)
        assert (g[lp + 1] == g[lp] + 1).all()
    for x, us in users.items():
        if len(us) > 1:
            for s, p in us:
                assert tr[s][p] == 0, "trainable token shared"
                # the copied context token before a trainable token is private
                assert not (p + 1 < len(seqs[s]) and tr[s][p + 1]), "join token shared"
    # pads
    for r in range(plan.n_rows):
        u = plan.used[r]
        assert (plan.token_ids[r, u:] == 0).all() and (plan.position_ids[r, u:] == 0).all()
        assert (plan.subtree_end[r, u:] == np.arange(u, T)).all()
        assert (plan.loss_mask[r, u:] == 0).all()
        assert u == plan.bins[r].token_count


def _check_visibility(plan, seqs):
    """The visible set of the query holding position p of sequence s is the
    set of row indices of positions 0..p of s (ancestors from parent
    pointers), and the interval predicate on subtree_end gives the same set."""
    T = plan.row_len
    offs = np.concatenate([[0], np.cumsum([len(s) for s in seqs])])
    trees = {}
    for s in range(len(seqs)):
        g = plan.gather_index[offs[s]:offs[s + 1]]
        r = int(g[0] // T)
        rt = trees.setdefault(r, RowTree(plan, r))
        cols = g % T
        se = plan.subtree_end[r]
        j = np.arange(T)
        for p in range(len(cols)):
            i = int(cols[p])
            want = cols[:p + 1]
            assert rt.visible(i).tolist() == want.tolist()
            pred = np.flatnonzero((j <= i) & (se >= i))
            assert pred.tolist() == want.tolist()


@pytest.mark.parametrize("seed", range(25))
def test_random_forest_layout_and_visibility(seed):
    ms = [1, 4, 64][seed % 3]
    b = W.random_forest(seed, n_roots=1 + seed % 3, min_shared=ms, len_lo=1,
                        len_hi=12 if ms < 64 else 90, row_len=600,
                        vocab=[4, 50, W.VOCAB][seed % 3], p_trainable_tail=0.3)
    plan = P.pack(b.seqs, b.trainable, b.row_len, ms, b.family)
    _check_layout(plan, b.seqs, b.trainable, ms)
    _check_visibility(plan, b.seqs)
    # Segment lengths obey the minimum: a shared segment is at least
    # min_shared - 1 long (the agreed run less the copied context token).
    shared = [sg for sg in plan.trie.segments if not sg.is_leaf]
    for sg in shared:
        assert sg.length >= ms - 1


@pytest.mark.parametrize("name", ["tiny", "grpo", "curriculum", "bushy"])
def test_config_layouts(name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    plan = P.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
    _check_layout(plan, b.seqs, b.trainable, b.min_shared)
    if name != "curriculum":
        assert plan.n_rows == 1


def test_useful_pairs_equal_sum_positions():
    from oracle.attn import useful_pairs
    b = W.tiny(0)
    plan = P.pack(b.seqs, b.trainable, b.row_len, 64)
    u = plan.used[0]
    assert useful_pairs(plan) == int((plan.position_ids[0, :u].astype(np.int64) + 1).sum())


# --- the appendix: union-size load is monotone submodular -----------------

@pytest.mark.parametrize("seed", range(10))
def test_bin_load_is_union_size_and_submodular(seed):
    b = W.random_forest(seed, n_roots=2, min_shared=4, len_lo=2, len_hi=20, row_len=10 ** 6)
    trie = P.build_trie(b.seqs, b.trainable, 4)
    leaves = P.make_leaves(trie)
    rng = np.random.default_rng(seed)
    order = rng.permutation(len(leaves))
    probe = leaves[int(order[-1])]
    bn = P.Bin()
    deltas = []
    for i in order[:-1]:
        deltas.append(bn.insertion_delta(probe))
        bn.add(leaves[int(i)])
        union = set()
        for lf in bn.leaves:
            union.update(sid for sid, _ in lf.segment_path)
        assert bn.token_count == sum(trie.segments[s].length for s in union)
    deltas.append(bn.insertion_delta(probe))
    assert all(a >= c for a, c in zip(deltas, deltas[1:]))


# --- edge cases ------------------------------------------------------------

def test_too_long_and_invalid():
    seqs, tr = _private_batch([5, 11])
    with pytest.raises(P.PackError) as e:
        P.pack(seqs, tr, 10, 64)
    assert e.value.kind == "ETOOLONG"
    with pytest.raises(P.PackError):
        P.pack([np.zeros(0, np.int32)], [np.zeros(0, np.uint8)], 10, 64)


def test_empty_batch():
    plan = P.pack([], [], 128, 64)
    assert plan.n_rows == 0 and plan.gather_index.size == 0


def test_identical_and_prefix_sequences():
    base = np.arange(100, 200, dtype=np.int32)
    seqs = [base.copy(), base.copy(), base[:80].copy()]
    tr = [np.zeros(100, np.uint8), np.zeros(100, np.uint8), np.zeros(80, np.uint8)]
    # min 16: all three share 80 tokens, the two long ones the next 20 as
    # well; the sequences that end inside a shared run get empty leaves
    plan = P.pack(seqs, tr, 1000, 16)
    assert plan.used == [100]
    _check_layout(plan, seqs, tr, 16)
    _check_visibility(plan, seqs)
    # min 64: the 20-token run after the split is too short and is duplicated
    plan = P.pack(seqs, tr, 1000, 64)
    assert plan.used == [80 + 20 + 20]
    # identical trainable completions are never merged
    tr2 = [np.array([0] * 70 + [1] * 30, np.uint8)] * 2
    plan2 = P.pack([base, base], tr2, 1000, 64)
    assert plan2.used == [69 + 2 * 31]


def test_short_run_pushed_down():
    """A shared run shorter than the minimum is not emitted; a long run below
    it is still shared within each sub-partition."""
    a = np.arange(0, 10, dtype=np.int32)
    x = np.arange(500, 600, dtype=np.int32)
    y = np.arange(700, 800, dtype=np.int32)
    seqs = [np.concatenate([a, [1], x]), np.concatenate([a, [1], x]), np.concatenate([a, [2], y])]
    tr = [np.zeros(len(s), np.uint8) for s in seqs]
    plan = P.pack(seqs, tr, 1000, 64)
    # seqs 0 and 1 share all 111 tokens; seq 2 duplicates the 10-token run
    assert plan.used == [111 + 111]
    _check_visibility(plan, seqs)


def test_per_family_trees_use_more_rows():
    b = W.curriculum(2)
    glob = P.pack(b.seqs, b.trainable, b.row_len, 64, b.family)
    per = P.pack(b.seqs, b.trainable, b.row_len, 64, b.family, per_family=True)
    assert per.n_rows >= glob.n_rows
    assert sum(per.used) >= sum(glob.used)
