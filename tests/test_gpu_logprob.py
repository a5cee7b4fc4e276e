"""Next-token log-probability gather on the GPU (stp_logprob_gather) against
the float64 oracle (oracle/logprob.py) on the same bf16 inputs.

Tolerance: the logits are bf16 products summed in float32 on the tensor cores
(D terms; the inputs give logits of spread about 2) and the log-sum-exp is
kept online in float32 with base-2 exponentials, so |logprob - oracle| stays
far below 1e-3 for D <= 4096; non-loss positions are exactly 0 and repeated
calls are bit-identical.
"""
import numpy as np
import pytest
import torch

from oracle import logprob as OL
from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _run(tok, mask, h, w):
    R, T = tok.shape
    desc = stp.logprob_desc(R, T, h.shape[1], w.shape[0])
    ws = torch.empty(stp.stp_logprob_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.full((R * T,), float("nan"), dtype=torch.float32, device="cuda")
    stp.stp_logprob_gather(desc, h.cuda(), w.cuda(), torch.from_numpy(np.ascontiguousarray(tok)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(mask)).cuda(), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), stp.stp_device_status(ws)


def _random_case(R, T, D, V, p_loss, seed):
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, V, size=(R, T), dtype=np.int32)
    mask = (rng.random((R, T)) < p_loss).astype(np.uint8)
    mask[:, -1] = 0
    h, w = W.logprob_tensors(R * T, D, V, seed=seed)
    return tok, mask, h, w


def _oracle(tok, mask, h, w):
    return OL.logprob_gather(tok, mask, h.float().numpy(), w.float().numpy())


@pytest.mark.parametrize("R,T,D,V,p", [
    (2, 256, 128, 1000, 0.5),      # ragged last vocabulary tile
    (1, 384, 64, 1, 0.3),          # a one-token vocabulary: every logprob is 0
    (1, 256, 64, 255, 0.9),        # vocabulary inside one tile
    (1, 256, 192, 257, 0.9),       # two tiles, the second holding one row
    (3, 128, 64, 64 * 256 + 3, 0.2),   # more tiles than splits: uneven split sizes
    (1, 512, 1024, 5000, 0.05),    # long hidden loop, sparse loss positions
])
def test_matches_oracle(R, T, D, V, p):
    tok, mask, h, w = _random_case(R, T, D, V, p, seed=R * 7 + T + D + V)
    got, status = _run(tok, mask, h, w)
    assert status == stp.STP_OK
    want = _oracle(tok, mask, h, w)
    m = mask.reshape(-1).astype(bool)
    assert np.all(got[~m] == 0.0)
    np.testing.assert_allclose(got[m], want[m], atol=TOL, rtol=0)


def test_tiles_without_loss_positions_and_empty_mask():
    tok, mask, h, w = _random_case(2, 512, 128, 700, 0.5, seed=11)
    mask[0, :] = 0
    mask[1, 128:384] = 0        # whole tiles without loss positions
    got, status = _run(tok, mask, h, w)
    assert status == stp.STP_OK
    np.testing.assert_allclose(got, _oracle(tok, mask, h, w), atol=TOL, rtol=0)
    mask[:] = 0
    got, status = _run(tok, mask, h, w)
    assert status == stp.STP_OK and np.all(got == 0.0)


def test_deterministic():
    tok, mask, h, w = _random_case(4, 256, 256, 3000, 0.6, seed=5)
    a, _ = _run(tok, mask, h, w)
    b, _ = _run(tok, mask, h, w)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_packed_forest_rows():
    """loss_mask and token ids straight from the packer (join copies in place)."""
    b = W.random_forest(3, n_roots=3, max_depth=3, max_children=3, len_lo=6, len_hi=60, row_len=512,
                        min_shared=8, vocab=97)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    R, T = plan.token_ids.shape
    h, w = W.logprob_tensors(R * T, 128, 97, seed=3)
    got, status = _run(plan.token_ids, plan.loss_mask, h, w)
    assert status == stp.STP_OK
    np.testing.assert_allclose(got, _oracle(plan.token_ids, plan.loss_mask, h, w), atol=TOL, rtol=0)


def test_bad_targets_set_the_device_error_word():
    tok, mask, h, w = _random_case(1, 256, 64, 300, 0.5, seed=2)
    m2 = mask.copy()
    m2[0, -1] = 1                       # a loss position at the end of its row
    _, status = _run(tok, m2, h, w)
    assert status == stp.STP_EDEVICE
    t2 = tok.copy()
    x = int(np.flatnonzero(mask[0])[0])
    t2[0, x + 1] = 300                  # a target outside the vocabulary
    _, status = _run(t2, mask, h, w)
    assert status == stp.STP_EDEVICE
    _, status = _run(tok, mask, h, w)   # the error word is cleared by the next call
    assert status == stp.STP_OK


def test_descriptor_checks():
    for bad in [stp.logprob_desc(1, 100, 64, 10), stp.logprob_desc(1, 128, 96, 10),
                stp.logprob_desc(1, 128, 64, 0), stp.logprob_desc(-1, 128, 64, 10)]:
        with pytest.raises(stp.StpError):
            stp.stp_logprob_workspace_size(bad)


def test_grpo_row_full_size_sampled():
    """The benchmarked launch: the GRPO row (16384 positions, loss mask and
    targets from the packer), hidden 4096, a 151936-token vocabulary; the
    oracle checks 48 sampled loss positions and the non-loss zeros."""
    b = W.grpo(seed=W.CONFIG_SEEDS["grpo"])
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    R, T = plan.token_ids.shape
    D, V = 4096, 151936
    h, w = W.logprob_tensors(R * T, D, V, seed=1)
    got, status = _run(plan.token_ids, plan.loss_mask, h, w)
    assert status == stp.STP_OK
    m = plan.loss_mask.reshape(-1).astype(bool)
    assert np.all(got[~m] == 0.0)
    xs = np.random.default_rng(0).choice(np.flatnonzero(m), 48, replace=False)
    tok = plan.token_ids.reshape(-1)
    # the oracle over the sampled positions only: each is its own one-position row pair
    sub_tok = np.stack([tok[xs], tok[xs + 1]], 1).astype(np.int32)
    sub_mask = np.zeros_like(sub_tok, dtype=np.uint8)
    sub_mask[:, 0] = 1
    hs = torch.zeros(2 * len(xs), D, dtype=torch.bfloat16)
    hs[0::2] = h[torch.from_numpy(xs)]
    want = OL.logprob_gather(sub_tok, sub_mask, hs.float().numpy(), w.float().numpy()).reshape(-1, 2)[:, 0]
    np.testing.assert_allclose(got[xs], want, atol=TOL, rtol=0)
