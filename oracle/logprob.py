"""Oracle: next-token log-probabilities gathered over packed rows, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source (prefix-tree-packing page, tree-build section on trainable tokens and
the join copy, and the materialization section): every trainable token's
predecessor sits immediately before it in the same packed row (the join copy
exists for exactly that), so the loss of a packed row is read off position x
for the token at x + 1 wherever loss_mask[x] = 1.

For a vocabulary projection W [V, D] and hidden states h [N, D] of the packed
positions (N = R * T):

    logits[x, v] = h[x] . W[v]
    logprob[x]   = logits[x, tok[x + 1]] - ln sum_v exp(logits[x, v])   if loss_mask[x]
                 = 0                                                      otherwise
"""
from __future__ import annotations

import numpy as np


def logprob_gather(token_ids: np.ndarray, loss_mask: np.ndarray, h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """token_ids, loss_mask [R, T]; h [R * T, D]; w [V, D] -> float64 [R * T]."""
    R, T = token_ids.shape
    tok = np.asarray(token_ids).reshape(-1)
    m = np.asarray(loss_mask).reshape(-1).astype(bool)
    out = np.zeros(R * T)
    xs = np.flatnonzero(m)
    if len(xs) == 0:
        return out
    if np.any(xs % T == T - 1):
        raise ValueError("a loss position is the last of its row")
    logits = np.asarray(h, np.float64)[xs] @ np.asarray(w, np.float64).T       # [n, V]
    mx = logits.max(1, keepdims=True)
    lse = (mx + np.log(np.exp(logits - mx).sum(1, keepdims=True)))[:, 0]
    out[xs] = logits[np.arange(len(xs)), tok[xs + 1]] - lse
    return out


def sequence_logprobs(seq: np.ndarray, trainable: np.ndarray, h_of, w: np.ndarray) -> np.ndarray:
    """The same quantity on one unpacked sequence: for every trainable token at
    position p >= 1, log p(seq[p] | hidden state of position p - 1); h_of(tok,
    pos) gives a hidden state from a token id and its position."""
    out = []
    for p in range(1, len(seq)):
        if trainable[p]:
            lg = np.asarray(w, np.float64) @ np.asarray(h_of(seq[p - 1], p - 1), np.float64)
            mx = lg.max()
            out.append(lg[seq[p]] - (mx + np.log(np.exp(lg - mx).sum())))
    return np.asarray(out)
