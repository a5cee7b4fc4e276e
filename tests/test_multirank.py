"""The multi-rank host logic on CPU: two gloo ranks (one process each).

Each rank packs its own batch (weak scaling), the unit shards of one batch
cover every (row, kv head) exactly once, and the only collective -- the
maximum of the step times -- returns the slowest rank's value everywhere.
"""
import os
import socket

import numpy as np
import pytest

from sft_trie_build_gb300.shard import row_useful_pairs, shard_units, shard_units_weighted, unit_runs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sft_trie_build_gb300 import stp
        from sft_trie_build_gb300 import workloads as W
        from sft_trie_build_gb300.shard import max_over_ranks, rank_seed

        b = W.grpo(rank_seed(W.CONFIG_SEEDS["grpo"], rank))
        tokens, offsets, train = b.flat()
        plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=64)
        info = stp.stp_plan_info(plan)
        se = stp.stp_plan_write(plan)["subtree_end"]
        # one multi-row batch split across ranks
        c = W.curriculum(2)
        ct, co, ctr = c.flat()
        cinfo = stp.stp_plan_info(stp.stp_pack(ct, co, ctr, c.family, row_len=c.row_len, min_shared=64))
        u0, u1 = shard_units(cinfo["n_rows"], 8, world, rank)
        shards = [None] * world
        dist.all_gather_object(shards, (u0, u1))
        cplan = stp.stp_pack(ct, co, ctr, c.family, row_len=c.row_len, min_shared=64)
        cmeta = stp.stp_plan_write(cplan)
        gi = cmeta["gather_index"]
        used = np.zeros(cinfo["n_rows"], np.int64)
        np.maximum.at(used, gi // c.row_len, gi % c.row_len + 1)
        work = row_useful_pairs(cmeta["position_ids"], used)
        wshards = [None] * world
        dist.all_gather_object(wshards, shard_units_weighted(work, 8, world, rank))
        t_max = max_over_ranks(10.0 + rank)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), se=se, seed=b.seed, pairs=info["useful_pairs"],
                 shards=np.array(shards), wshards=np.array(wshards), n_rows=cinfo["n_rows"], t_max=t_max)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(stp_lib, tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    # weak scaling: different batches, each packed on its own rank
    assert int(r0["seed"]) != int(r1["seed"])
    assert not np.array_equal(r0["se"], r1["se"])
    # the max-over-ranks timing is the slowest rank's, on every rank
    assert float(r0["t_max"]) == float(r1["t_max"]) == 11.0
    # the shards of one batch partition its units
    shards = r0["shards"]
    assert np.array_equal(shards, r1["shards"])
    n_units = int(r0["n_rows"]) * 8
    for sh in (shards, r0["wshards"]):
        covered = np.zeros(n_units, int)
        for u0, u1 in sh:
            covered[u0:u1] += 1
        assert (covered == 1).all()
    assert np.array_equal(r0["wshards"], r1["wshards"])


@pytest.mark.parametrize("rows,heads,world", [(1, 8, 2), (28, 8, 3), (5, 3, 4), (2, 1, 4)])
def test_shard_units_partition(rows, heads, world):
    seen = np.zeros(rows * heads, int)
    sizes = []
    for rank in range(world):
        u0, u1 = shard_units(rows, heads, world, rank)
        sizes.append(u1 - u0)
        for r, g0, g1 in unit_runs(u0, u1, heads):
            assert 0 <= r < rows and 0 <= g0 < g1 <= heads
            seen[r * heads + g0: r * heads + g1] += 1
    assert (seen == 1).all()
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("world", [2, 3, 4, 7])
def test_weighted_shards_balance_work(stp_lib, world):
    """On the global-tree batch (28 rows of very different work), work-weighted
    shards partition the units, each rank's work stays within one unit's
    weight of the mean, and the busiest rank carries no more than with
    equal-count shards.  The work of a row is checked against the packer's
    own count (stp_plan_info)."""
    from sft_trie_build_gb300 import stp
    from sft_trie_build_gb300 import workloads as W

    c = W.curriculum(W.CONFIG_SEEDS["curriculum"])
    t, o, tr = c.flat()
    plan = stp.stp_pack(t, o, tr, c.family, row_len=c.row_len, min_shared=64)
    info = stp.stp_plan_info(plan)
    meta = stp.stp_plan_write(plan)
    gi = meta["gather_index"]
    R, H = info["n_rows"], 8
    used = np.zeros(R, np.int64)
    np.maximum.at(used, gi // c.row_len, gi % c.row_len + 1)
    work = row_useful_pairs(meta["position_ids"], used)
    assert int(work.sum()) == info["useful_pairs"]
    unit_w = np.repeat(work, H)
    covered = np.zeros(R * H, int)
    wmax, cmax = 0, 0
    for rank in range(world):
        u0, u1 = shard_units_weighted(work, H, world, rank)
        covered[u0:u1] += 1
        wmax = max(wmax, unit_w[u0:u1].sum())
        a, b = shard_units(R, H, world, rank)
        cmax = max(cmax, unit_w[a:b].sum())
    assert (covered == 1).all()
    assert wmax <= unit_w.sum() / world + unit_w.max()
    assert wmax <= cmax
