"""Tree-aware Gated DeltaNet forward on the GPU (stp_gdn_fwd) against the
float64 oracle (oracle/gdn.py) on the same inputs (x rounded to bf16).

Tolerance: the path convolution and the normalization run in float32, but
q, k, v and every per-chunk tensor-core operand (W, Q~, K~, P, the state and
V') are rounded to bf16 (relative 2^-9) with float32 sums, and the state is
carried in float32 from chunk to chunk; so max |o - oracle| <= 2e-2 max |o|
and the mean error <= 2e-3 max |o|.  Pads give exactly 0 and repeated calls
are bit-identical.
"""
import numpy as np
import pytest

from gdn_helpers import oracle_rows, oracle_sequence_heads, run_gdn
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _compare(po, H, seed=1):
    outs, status, inputs, scale = run_gdn(po, H, seed=seed, reps=2)
    assert status == 0
    o = outs[0]
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    ref = oracle_rows(po, H, inputs, scale)
    T = po.row_len
    real = np.concatenate([np.arange(r * T, r * T + po.used[r]) for r in range(po.n_rows)])
    pads = np.setdiff1d(np.arange(len(o)), real)
    assert np.all(o[pads] == 0.0)
    scale_ref = np.abs(ref[real]).max()
    d = np.abs(o[real] - ref[real])
    assert d.max() <= 2e-2 * scale_ref, (d.max(), scale_ref)
    assert d.mean() <= 2e-3 * scale_ref, (d.mean(), scale_ref)


@pytest.mark.parametrize("seed", range(3))
def test_random_forests(seed):
    """Single-token segments, ragged chunks, forks at every depth, pads."""
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=1, len_hi=150, row_len=512,
                        min_shared=4, vocab=41)
    _compare(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared), H=2, seed=seed)


@pytest.mark.parametrize("T,seed", [(200, 0), (456, 12)])
def test_rows_not_multiple_of_block(T, seed):
    """Rows whose length is not a multiple of the convolution's token block:
    some blocks start in one row's pads and hold the next row's first tokens
    (they must be copied), others lie in one row's pads (they need not be).
    Both kinds occur in these two batches for blocks of 64 and of 128."""
    b = W.random_forest(seed, n_roots=6, max_depth=2, max_children=3, len_lo=5, len_hi=60, row_len=T,
                        min_shared=4, vocab=41)
    po = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    N = po.n_rows * T
    for blk in (64, 128):
        kinds = set()
        for x0 in range(0, N, blk):
            x1 = min(x0 + blk - 1, N - 1)
            if x0 % T >= po.used[x0 // T]:   # starts with a pad
                kinds.add("one row" if x0 // T == x1 // T else "straddles")
        assert kinds == {"one row", "straddles"}
    _compare(po, H=2, seed=seed)


def test_deep_narrow_tree():
    b = W.random_forest(11, n_roots=1, max_depth=6, max_children=2, len_lo=20, len_hi=90, row_len=1024,
                        min_shared=4, vocab=41)
    _compare(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared), H=1, seed=4)


def test_long_chain_many_chunks():
    rng = np.random.default_rng(5)
    seq = rng.integers(1, 1000, 1000).astype(np.int32)
    po = OP.pack([seq], [np.zeros(1000, np.uint8)], 1024, 64)
    _compare(po, H=2, seed=5)


def test_long_chain_cut_into_two_segments():
    """A 2200-token chain: the planner cuts it after 16 chunks (1024 + 1176
    tokens, the second segment the first's only child), so the state crosses
    one segment boundary through memory; every element against the oracle."""
    rng = np.random.default_rng(6)
    seq = rng.integers(1, 1000, 2200).astype(np.int32)
    _compare(OP.pack([seq], [np.zeros(2200, np.uint8)], 2304, 64), H=1, seed=6)


def test_tiny_workload():
    b = W.tiny(0)
    _compare(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared), H=3, seed=2)


def test_grpo_row_sampled():
    """The benchmarked shape: the GRPO row (a 5000-token prefix forked into 16
    rollouts), 16 heads of 128; two rollouts, unpacked, on two heads each."""
    b = W.grpo(seed=W.CONFIG_SEEDS["grpo"])
    po = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    H = 16
    outs, status, inputs, scale = run_gdn(po, H, seed=0)
    assert status == 0
    o = outs[0]
    offs = np.concatenate([[0], np.cumsum([len(s) for s in b.seqs])])
    for s, heads in ((0, (0, 7)), (9, (3, 15))):
        want, idx = oracle_sequence_heads(po, s, offs, heads, inputs, scale)
        got = o[idx][:, list(heads)]
        m = np.abs(want).max()
        d = np.abs(got - want)
        assert d.max() <= 2e-2 * m and d.mean() <= 2e-3 * m, (d.max(), d.mean(), m)
