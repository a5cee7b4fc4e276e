"""Pins of the logprob oracle (oracle/logprob.py): closed forms (a uniform
vocabulary, two-token logits), and the packed gather equal to per-sequence
log-probabilities on the unpacked sequences under a synthetic model whose
hidden state depends only on (token, position) -- which ties loss_mask, the
join copies and the gather index of the packer to the plain definition."""
import numpy as np
import pytest

from oracle import logprob as OL
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W


def test_uniform_vocabulary_is_minus_log_v():
    tok = np.array([[1, 2, 3, 0]], np.int32)
    mask = np.array([[1, 1, 0, 0]], np.uint8)
    h = np.zeros((4, 8))
    w = np.random.default_rng(0).standard_normal((50, 8))
    lp = OL.logprob_gather(tok, mask, h, w)
    np.testing.assert_allclose(lp, [-np.log(50), -np.log(50), 0, 0])


def test_two_token_vocabulary_is_log_sigmoid():
    tok = np.array([[0, 1, 0]], np.int32)
    mask = np.array([[1, 1, 0]], np.uint8)
    h = np.array([[2.0], [-0.5], [0.0]])
    w = np.array([[0.0], [1.0]])          # logits (0, h)
    lp = OL.logprob_gather(tok, mask, h, w)
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))  # noqa: E731
    np.testing.assert_allclose(lp[:2], [np.log(sig(2.0)), np.log(1.0 - sig(-0.5))])


def test_loss_at_row_end_is_rejected():
    with pytest.raises(ValueError):
        OL.logprob_gather(np.zeros((1, 3), np.int32), np.array([[0, 0, 1]], np.uint8), np.zeros((3, 2)),
                          np.zeros((4, 2)))


@pytest.mark.parametrize("seed", range(4))
def test_packed_gather_equals_unpacked_sequences(seed):
    """Random trees with trainable leaves (join copies included): the packed
    log-probabilities, gathered back per sequence through gather_index, equal
    the log-probabilities computed on each unpacked sequence."""
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=6, len_hi=60, row_len=512,
                        min_shared=8, vocab=97)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(seed)
    D, V = 16, 97
    E, P = rng.standard_normal((V, D)), rng.standard_normal((b.row_len, D)) * 0.3
    w = rng.standard_normal((V, D))
    h_of = lambda t, p: E[t] + P[p]  # noqa: E731
    tok, pos = plan.token_ids, plan.position_ids
    h = E[tok.reshape(-1)] + P[pos.reshape(-1)]
    lp = OL.logprob_gather(tok, plan.loss_mask, h, w)
    offs = np.concatenate([[0], np.cumsum([len(s) for s in b.seqs])])
    n_loss = 0
    for s, (seq, tr) in enumerate(zip(b.seqs, b.trainable)):
        want = OL.sequence_logprobs(seq, tr, h_of, w)
        flat = plan.gather_index[offs[s]: offs[s + 1]]
        got = [lp[flat[p - 1]] for p in range(1, len(seq)) if tr[p]]
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
        n_loss += len(want)
    assert n_loss > 0 and n_loss == int(plan.loss_mask.sum())   # no loss position left unaccounted
