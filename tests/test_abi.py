"""C ABI on the CPU: the library loads and exports every symbol stp.h declares,
and the C++ host packer matches the oracle bit for bit."""
import os
import re

import numpy as np
import pytest

from conftest import ROOT, golden
from oracle import attn as OA
from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W


def test_exports_every_declared_symbol(stp_lib):
    hdr = open(os.path.join(ROOT, "include", "stp.h")).read()
    declared = set(re.findall(r"\b(stp_[a-z_]+)\s*\(", hdr))
    assert declared == set(stp.EXPORTED)
    L = stp.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert "sm_103a" in stp.stp_version()


def _c_pack(b, flags=stp.STP_GLOBAL, row_len=None, min_shared=None):
    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=row_len or b.row_len,
                        min_shared=min_shared or b.min_shared, flags=flags)
    return plan, stp.stp_plan_write(plan), stp.stp_plan_info(plan)


def _assert_same(b, flags=stp.STP_GLOBAL, row_len=None, min_shared=None):
    row_len = row_len or b.row_len
    ms = min_shared or b.min_shared
    ref = OP.pack(b.seqs, b.trainable, row_len, ms, b.family,
                  per_family=bool(flags & stp.STP_PER_FAMILY), in_order=bool(flags & stp.STP_IN_ORDER))
    plan, out, info = _c_pack(b, flags, row_len, ms)
    assert info["n_rows"] == ref.n_rows
    for key in ("token_ids", "position_ids", "subtree_end", "loss_mask"):
        np.testing.assert_array_equal(out[key], getattr(ref, key), err_msg=key)
    np.testing.assert_array_equal(out["gather_index"], ref.gather_index)
    rows = stp.stp_plan_rows_of(plan)
    want = np.empty(len(b.seqs), np.int32)
    for r, bn in enumerate(ref.bins):
        for lf in bn.leaves:
            want[lf.seq] = r
    np.testing.assert_array_equal(rows, want)
    ri = OP.plan_info(ref)
    for k in ("n_rows", "row_len", "input_tokens", "packed_tokens", "n_segments", "n_leaves"):
        assert info[k] == ri[k], k
    assert info["tree_token_ratio"] == pytest.approx(ri["tree_token_ratio"], rel=1e-12)
    pos = ref.position_ids.astype(np.int64)
    useful = sum(int((pos[r, :u] + 1).sum()) for r, u in enumerate(ref.used))
    assert info["useful_pairs"] == useful
    return ref, out, info


@pytest.mark.parametrize("name", ["tiny", "grpo", "curriculum", "deep", "bushy"])
def test_packer_matches_oracle_on_workloads(stp_lib, name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    _assert_same(b)


@pytest.mark.parametrize("flags", [stp.STP_PER_FAMILY, stp.STP_IN_ORDER,
                                   stp.STP_PER_FAMILY | stp.STP_IN_ORDER])
def test_packer_flags_match_oracle(stp_lib, flags):
    _assert_same(W.curriculum(2), flags)


def test_packer_rollout32(stp_lib):
    g = golden("rollout32.json")
    b = W.rollout32(0)
    ref, out, info = _assert_same(b)
    assert ref.used == g["global_used"]
    _, _, info2 = _c_pack(b, stp.STP_IN_ORDER)
    assert info2["n_rows"] == 3 and info2["packed_tokens"] == sum(g["in_order_used"])


def test_packer_mask9(stp_lib):
    g = golden("mask9.json")
    seqs = [np.array(s, np.int32) for s in g["seqs"]]
    b = W.SeqBatch(seqs, [np.zeros(len(s), np.uint8) for s in seqs], None, g["row_len"], g["min_shared"])
    _, out, _ = _c_pack(b)
    assert out["subtree_end"][0].tolist() == g["subtree_end"]


@pytest.mark.parametrize("case", golden("bfd_small.json")["cases"], ids=lambda c: c["name"])
def test_packer_bfd_hand_worked(stp_lib, case):
    seqs = [np.arange(1000 * (i + 1), 1000 * (i + 1) + n, dtype=np.int32) for i, n in enumerate(case["sizes"])]
    fam = None if case["family"] is None else np.array(case["family"], np.int32)
    b = W.SeqBatch(seqs, [np.ones(len(s), np.uint8) for s in seqs], fam, case["row_len"], 64)
    plan, out, info = _c_pack(b)
    rows = stp.stp_plan_rows_of(plan)
    got = [sorted(np.flatnonzero(rows == r).tolist()) for r in range(info["n_rows"])]
    assert got == case["bins"]


@pytest.mark.parametrize("seed", range(40))
def test_packer_random_forests(stp_lib, seed):
    ms = [1, 2, 4, 16, 64][seed % 5]
    b = W.random_forest(seed, n_roots=1 + seed % 4, max_depth=1 + seed % 4, max_children=1 + seed % 5,
                        min_shared=ms, len_lo=1, len_hi=[6, 20, 90][seed % 3], row_len=[300, 700, 5000][seed % 3],
                        vocab=[3, 50, W.VOCAB][seed % 3], p_trainable_tail=0.3 if seed % 2 else 0.0,
                        p_nt_leaf=0.3)
    try:
        _assert_same(b)
    except OP.PackError as e:
        assert e.kind == "ETOOLONG"
        with pytest.raises(stp.StpError) as ei:
            _c_pack(b)
        assert ei.value.status == stp.STP_ETOOLONG
    if b.family is not None:
        try:
            _assert_same(b, stp.STP_PER_FAMILY)
        except OP.PackError:
            pass


def test_packer_no_trainable_mask_and_no_family(stp_lib):
    b = W.random_forest(3, n_roots=2, min_shared=2, len_hi=10, row_len=400, vocab=4)
    tokens, offsets, _ = b.flat()
    plan = stp.stp_pack(tokens, offsets, None, None, row_len=400, min_shared=2)
    out = stp.stp_plan_write(plan)
    ref = OP.pack(b.seqs, [np.zeros(len(s), np.uint8) for s in b.seqs], 400, 2, None)
    np.testing.assert_array_equal(out["subtree_end"], ref.subtree_end)
    np.testing.assert_array_equal(out["gather_index"], ref.gather_index)


def test_packer_errors(stp_lib):
    tok = np.arange(30, dtype=np.int32)
    with pytest.raises(stp.StpError) as e:
        stp.stp_pack(tok, np.array([0, 10, 30]), None, None, row_len=15)
    assert e.value.status == stp.STP_ETOOLONG
    with pytest.raises(stp.StpError) as e:
        stp.stp_pack(tok, np.array([0, 10, 10, 30]), None, None, row_len=64)
    assert e.value.status == stp.STP_EINVAL
    with pytest.raises(stp.StpError) as e:
        stp.stp_pack(tok, np.array([0, 30]), None, None, row_len=64, min_shared=0)
    assert e.value.status == stp.STP_EINVAL
    with pytest.raises(stp.StpError) as e:
        stp.stp_pack(tok, np.array([0, 30]), None, None, row_len=64, flags=8)
    assert e.value.status == stp.STP_EINVAL
    plan = stp.stp_pack(np.zeros(0, np.int32), np.array([0]), None, None, row_len=128)
    assert stp.stp_plan_info(plan)["n_rows"] == 0


def test_workspace_sizes_and_descriptor_checks(stp_lib):
    d = stp.Desc(2, 1024, 8, 2, 128, stp.STP_BF16)
    meta, fwd, bwd = stp.stp_workspace_size(d)
    nt = 1024 // 128
    assert meta >= 2 * nt * nt * (1 + 4 + 4) and fwd >= 4
    assert bwd >= 2 * 8 * 1024 * 4 + 2 * 1024 * 8 * 128 * 4
    for bad, code in ((stp.Desc(1, 1000, 8, 2, 128), stp.STP_EUNSUPPORTED),
                      (stp.Desc(1, 1024, 8, 3, 128), stp.STP_EUNSUPPORTED),
                      (stp.Desc(1, 1024, 8, 2, 64, stp.STP_BF16), stp.STP_EUNSUPPORTED),
                      (stp.Desc(1, 1024, 8, 2, 96, stp.STP_FP32), stp.STP_EUNSUPPORTED),
                      (stp.Desc(-1, 1024, 8, 2, 128), stp.STP_EINVAL)):
        with pytest.raises(stp.StpError) as e:
            stp.stp_workspace_size(bad)
        assert e.value.status == code
    stp.stp_workspace_size(stp.Desc(1, 256, 1, 1, 64, stp.STP_FP32))
    with pytest.raises(stp.StpError) as e:
        stp.stp_workspace_size(stp.Desc(1, 1024, 8, 2, 128, stp.STP_BF16, ds_groups=-1))
    assert e.value.status == stp.STP_EINVAL


def test_bwd_workspace_bounded_by_groups_held(stp_lib):
    """The dS part of the bf16 backward workspace scales with the kv-head
    groups held at once (ds_groups), not with Hq: the deep 32K-row shape
    (64 / 8 heads, 17605 tile pairs) needs 36.9 GB with every group's tiles
    held, 4.6 GB per group."""
    pairs, tile = 17605, 128 * 128 * 2
    full = stp.stp_workspace_size(stp.Desc(1, 32768, 64, 8, 128, stp.STP_BF16, 0.0, pairs))[2]
    per_group = pairs * 8 * tile
    assert full >= 8 * per_group
    for k in (1, 2, 4, 8, 100):
        ws = stp.stp_workspace_size(stp.Desc(1, 32768, 64, 8, 128, stp.STP_BF16, 0.0, pairs, ds_groups=k))[2]
        assert ws - full == (min(k, 8) - 8) * per_group
    # more kv heads than groups: group i holds kv heads [i Hkv / 8, (i + 1) Hkv / 8)
    a = stp.stp_workspace_size(stp.Desc(1, 1024, 32, 16, 128, stp.STP_BF16, 0.0, 10, ds_groups=1))[2]
    b = stp.stp_workspace_size(stp.Desc(1, 1024, 32, 16, 128, stp.STP_BF16, 0.0, 10, ds_groups=2))[2]
    assert b - a == 10 * 2 * 2 * tile


def test_useful_pairs_match_oracle_visible_sets(stp_lib):
    b = W.tiny(0)
    plan, _, info = _c_pack(b)
    ref = OP.pack(b.seqs, b.trainable, b.row_len, 64)
    assert info["useful_pairs"] == OA.useful_pairs(ref)


@pytest.mark.parametrize("name", ["tiny", "grpo", "curriculum", "deep", "bushy"])
def test_count_tile_pairs_matches_oracle_classes(stp_lib, name):
    """The host count of non-empty tile pairs equals the number of non-EMPTY
    entries of the oracle's tile-class matrix."""
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=b.min_shared)
    se = stp.stp_plan_write(plan)["subtree_end"]
    ref = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
    assert stp.stp_count_tile_pairs(se) == int((OA.tile_classes(ref) != OA.EMPTY).sum())


def test_count_tile_pairs_edge_cases(stp_lib):
    T = 256
    diag = np.arange(T, dtype=np.int32)[None]          # every token sees itself only
    assert stp.stp_count_tile_pairs(diag) == 2
    full = np.full((1, T), T - 1, dtype=np.int32)      # causal over the whole row
    assert stp.stp_count_tile_pairs(full) == 3
    assert stp.stp_count_tile_pairs(np.zeros((0, T), np.int32)) == 0
    bad = diag.copy()
    bad[0, 10] = 5
    with pytest.raises(stp.StpError) as e:
        stp.stp_count_tile_pairs(bad)
    assert e.value.status == stp.STP_EINVAL
    with pytest.raises(stp.StpError):
        stp.stp_count_tile_pairs(np.zeros((1, 100), np.int32))
