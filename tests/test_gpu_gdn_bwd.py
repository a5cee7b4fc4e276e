"""Gated DeltaNet backward on the GPU (stp_gdn_fwd_train + stp_gdn_bwd)
against the float64 oracle's reverse mode (oracle.gdn.gdn_row_grads) on the
same inputs, for L = sum dO . o with dO ~ N(0, 1) on real tokens.

Tolerance: every product of the backward takes bf16 operands (relative
rounding 2^-9 = 2e-3) with float32 sums, on top of the forward's bf16 chunk
operands; a gradient passes through at most three such roundings in a chain
(e.g. dS_n -> dV' -> dW -> dT -> dA -> dk), each adding about 2e-3 of its
input's scale, so the error stays within 2e-2 of the gradient's largest
magnitude (mean within 2e-3), the bar of the forward.  Observed on the GRPO
row: at most 5.8e-3 (max) and 6.6e-4 (mean).  Pads get exactly 0.
"""
import numpy as np
import pytest

from gdn_helpers import oracle_row_grads, run_gdn_train
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _compare(po, H, seed):
    outs, status, inputs, dO, scale = run_gdn_train(po, H, seed)
    assert status == 0
    _, dx, dw, dg, db = outs
    want = oracle_row_grads(po, H, inputs, dO, scale)
    T = po.row_len
    real = np.concatenate([np.arange(r * T, r * T + po.used[r]) for r in range(po.n_rows)])
    pads = np.setdiff1d(np.arange(po.n_rows * T), real)
    assert np.all(dx[pads] == 0) and np.all(dg[pads] == 0) and np.all(db[pads] == 0)
    for name, got, ref in (("dx", dx[real], want[0][real]), ("dconv_w", dw, want[1]),
                           ("dg", dg[real], want[2][real]), ("dbeta", db[real], want[3][real])):
        m = np.abs(ref).max()
        d = np.abs(got - ref)
        print(name, float(d.max() / m), float(d.mean() / m))
        assert d.max() <= 2e-2 * m and d.mean() <= 2e-3 * m, (name, d.max(), d.mean(), m)


@pytest.mark.parametrize("seed", range(2))
def test_random_forests(seed):
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=1, len_hi=150, row_len=512,
                        min_shared=4, vocab=41)
    _compare(OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared), H=2, seed=seed)


def test_long_chain_many_chunks():
    rng = np.random.default_rng(5)
    seq = rng.integers(1, 1000, 700).astype(np.int32)
    _compare(OP.pack([seq], [np.zeros(700, np.uint8)], 768, 64), H=1, seed=5)


def test_grpo_row_two_heads():
    """The benchmarked shape, every element of two heads: the GRPO row (a
    5000-token prefix, 79 chunks walked one after another, forked into 16
    rollouts), 16 heads of 128.  Heads never mix in the layer core, so the
    oracle of head h is the layer with one head on h's q, k, v channels."""
    from gdn_helpers import oracle_head_grads

    b = W.grpo(seed=W.CONFIG_SEEDS["grpo"])
    po = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    H = 16
    outs, status, inputs, dO, scale = run_gdn_train(po, H, seed=0)
    assert status == 0
    _, dx, dw, dg, db = outs
    real = np.arange(po.used[0])
    errs = {}
    for h, (ch, gx, gw, gg, gb) in oracle_head_grads(po, 0, inputs, dO, scale, H, (0, 9)).items():
        for name, got, ref in (("dx", dx[real][:, ch], gx[real]), ("dconv_w", dw[ch], gw),
                               ("dg", dg[real, h], gg[real]), ("dbeta", db[real, h], gb[real])):
            m = np.abs(ref).max()
            d = np.abs(got - ref)
            errs[(h, name)] = (float(d.max() / m), float(d.mean() / m))
            assert d.max() <= 2e-2 * m and d.mean() <= 2e-3 * m, (h, name, d.max(), d.mean(), m)
    print("\nGRPO row GDN backward, max / mean error relative to max |oracle|:", errs)


def test_repeat_bit_identical():
    """Every gradient is summed in one fixed order: two backward calls on the
    same inputs give the same bits."""
    b = W.random_forest(3, n_roots=3, max_depth=3, max_children=3, len_lo=1, len_hi=150, row_len=512,
                        min_shared=4, vocab=41)
    po = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    a = run_gdn_train(po, 2, seed=3)[0]
    c = run_gdn_train(po, 2, seed=3)[0]
    for x, y in zip(a, c):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
