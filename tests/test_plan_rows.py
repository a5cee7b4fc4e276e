"""'What if' planning (stp_plan_rows, stp_plan_rows_many): the rows and packed
tokens of a candidate batch drawn from a pool, without a plan or rows.  The
counts must equal those of packing that batch, checked against the oracle's
own pack of the same sequences (bit-exact integers) and against stp_pack."""
import numpy as np
import pytest

from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W


def _pool(name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    tokens, offsets, train = b.flat()
    return b, tokens, offsets, train


@pytest.mark.parametrize("name", ["tiny", "grpo", "curriculum", "bushy"])
@pytest.mark.parametrize("flags", [stp.STP_GLOBAL, stp.STP_PER_FAMILY, stp.STP_IN_ORDER])
def test_whole_pool_equals_pack(stp_lib, name, flags):
    b, t, o, tr = _pool(name)
    rows, packed = stp.stp_plan_rows(t, o, tr, b.family, row_len=b.row_len, min_shared=b.min_shared, flags=flags)
    info = stp.stp_plan_info(stp.stp_pack(t, o, tr, b.family, row_len=b.row_len, min_shared=b.min_shared,
                                          flags=flags))
    assert (rows, packed) == (info["n_rows"], info["packed_tokens"])


@pytest.mark.parametrize("flags", [stp.STP_GLOBAL, stp.STP_PER_FAMILY, stp.STP_IN_ORDER])
def test_subsets_match_oracle(stp_lib, flags):
    """Random candidate batches of the curriculum pool (whole groups and loose
    sequences, in a shuffled order) against the oracle packing them."""
    b, t, o, tr = _pool("curriculum")
    n = len(b.seqs)
    rng = np.random.default_rng(7)
    fam = np.asarray(b.family)
    subsets = []
    for k in range(4):
        groups = rng.choice(np.unique(fam), size=3 + k, replace=False)
        idx = np.flatnonzero(np.isin(fam, groups))
        extra = rng.choice(n, size=5, replace=False)
        sub = np.concatenate([idx, extra]).astype(np.int32)
        rng.shuffle(sub)
        subsets.append(sub)
    rows, packed = stp.stp_plan_rows_many(t, o, tr, b.family, subsets, row_len=b.row_len,
                                          min_shared=b.min_shared, flags=flags, n_threads=3)
    for sub, r, p in zip(subsets, rows, packed):
        ref = OP.pack([b.seqs[i] for i in sub], [b.trainable[i] for i in sub], b.row_len, b.min_shared,
                      [b.family[i] for i in sub], per_family=bool(flags & stp.STP_PER_FAMILY),
                      in_order=bool(flags & stp.STP_IN_ORDER))
        info = OP.plan_info(ref)
        assert (int(r), int(p)) == (info["n_rows"], info["packed_tokens"])
        assert (int(r), int(p)) == stp.stp_plan_rows(t, o, tr, b.family, sub, row_len=b.row_len,
                                                     min_shared=b.min_shared, flags=flags)


@pytest.mark.parametrize("seed", range(4))
def test_random_forest_subsets_with_repeats(stp_lib, seed):
    """Index lists with repeats and any order, on random trees."""
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=8, len_hi=120, row_len=1024,
                        min_shared=16, vocab=W.VOCAB)
    t, o, tr = b.flat()
    rng = np.random.default_rng(seed)
    sub = rng.integers(0, len(b.seqs), size=2 * len(b.seqs)).astype(np.int32)
    r, p = stp.stp_plan_rows(t, o, tr, b.family, sub, row_len=b.row_len, min_shared=b.min_shared)
    ref = OP.plan_info(OP.pack([b.seqs[i] for i in sub], [b.trainable[i] for i in sub], b.row_len,
                               b.min_shared, None if b.family is None else [b.family[i] for i in sub]))
    assert (r, p) == (ref["n_rows"], ref["packed_tokens"])


def test_many_equals_single_any_thread_count(stp_lib):
    b, t, o, tr = _pool("bushy")
    rng = np.random.default_rng(1)
    subs = [rng.choice(len(b.seqs), size=int(rng.integers(1, len(b.seqs))), replace=False) for _ in range(12)]
    single = [stp.stp_plan_rows(t, o, tr, b.family, s, row_len=b.row_len) for s in subs]
    for nt in (1, 4, 0):
        rows, packed = stp.stp_plan_rows_many(t, o, tr, b.family, subs, row_len=b.row_len, n_threads=nt)
        assert [(int(r), int(p)) for r, p in zip(rows, packed)] == single


def test_errors(stp_lib):
    b, t, o, tr = _pool("tiny")
    n = len(b.seqs)
    with pytest.raises(stp.StpError) as e:
        stp.stp_plan_rows(t, o, tr, b.family, [0, n], row_len=b.row_len)
    assert e.value.status == stp.STP_EINVAL
    with pytest.raises(stp.StpError) as e:
        stp.stp_plan_rows_many(t, o, tr, b.family, [[0], [1], [0, -1]], row_len=b.row_len)
    assert e.value.status == stp.STP_EINVAL and "subset 2" in str(e.value)
    with pytest.raises(stp.StpError) as e:
        stp.stp_plan_rows(t, o, tr, b.family, [0], row_len=8)
    assert e.value.status == stp.STP_ETOOLONG
    assert stp.stp_plan_rows(t, o, tr, b.family, [], row_len=b.row_len) == (0, 0)
    rows, packed = stp.stp_plan_rows_many(t, o, tr, b.family, [], row_len=b.row_len)
    assert len(rows) == 0 and len(packed) == 0


def test_plan_times_are_reported(stp_lib):
    """stp_plan_times gives the walk and placement times of the plan's own
    stp_pack call: non-negative, and the placement of a many-group batch is
    measurable."""
    b = W.curriculum(W.CONFIG_SEEDS["curriculum"])
    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=b.min_shared)
    t = stp.stp_plan_times(plan)
    assert t["walk_ms"] >= 0.0 and t["place_ms"] >= 0.0
    assert t["walk_ms"] + t["place_ms"] > 0.0
