"""Oracle: the Gated DeltaNet layer core over packed prefix trees, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source (prefix-tree-packing page, GDN section; ART-Optimized Megatron page,
the Gated DeltaNet paragraphs): GDN carries a running state from token to
token; on a packed tree the state is threaded along each token's own path,
forked at every branch point (a child starts from its parent's final state)
and reset to zero at every root, and the short causal convolution in front
of the recurrence reads the previous tokens of the same path (the parent's
last inputs are handed to each child).  The packed result must equal the
layer run on every sequence unpacked.

The layer core, per head h (state S of shape [d_k, d_v]):

    y_t        = SiLU(sum_{i=0..3} w[:, i] * x_{t-3+i})      (path order, zero before the root)
    q, k, v    = the three channel blocks of y_t, split into heads of d
    q, k      <- q / sqrt(|q|^2 + eps), k / sqrt(|k|^2 + eps)        (eps = 1e-6)
    alpha_t    = exp(g_t)
    S_t        = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T
    o_t        = scale * S_t^T q_t

(the gated delta rule: decay the state, then move the value stored under
k_t a fraction beta_t of the way toward v_t).

Paths come from the packer's parent pointers (``oracle.attn.RowTree``),
never from ``subtree_end``: the token before i on its path is the last
visible key before i.  A pad sees only itself and is its own root.
"""
from __future__ import annotations

import numpy as np

from .attn import RowTree
from .pack import Plan

EPS = 1e-6
WIDTH = 4


def silu(z):
    return z / (1.0 + np.exp(-z))


def l2norm(z):
    return z / np.sqrt((z * z).sum(-1, keepdims=True) + EPS)


def path_prev(plan: Plan, r: int) -> np.ndarray:
    """int64 [T]: the token before i on its path, -1 at a root or a pad."""
    rt = RowTree(plan, r)
    prev = np.full(plan.row_len, -1, np.int64)
    for i in range(plan.row_len):
        vis = rt.visible(i)
        if len(vis) > 1:
            prev[i] = vis[-2]
    return prev


def conv_path(x: np.ndarray, conv_w: np.ndarray, prev: np.ndarray) -> np.ndarray:
    """y [T, C] = SiLU of the width-4 causal depthwise convolution along each
    token's path (tap 3 = the token itself, tap 0 = three tokens back)."""
    T, C = x.shape
    y = np.zeros((T, C))
    for t in range(T):
        acc = np.zeros(C)
        j = t
        for i in range(WIDTH - 1, -1, -1):
            if j < 0:
                break
            acc += conv_w[:, i] * x[j]
            j = prev[j]
        y[t] = silu(acc)
    return y


def split_heads(y: np.ndarray, H: int, d: int):
    """(q, k, v) [T, H, d] from the channel blocks of y, q and k normalized."""
    T = y.shape[0]
    q = y[:, 0 * H * d: 1 * H * d].reshape(T, H, d)
    k = y[:, 1 * H * d: 2 * H * d].reshape(T, H, d)
    v = y[:, 2 * H * d: 3 * H * d].reshape(T, H, d)
    return l2norm(q), l2norm(k), v


def delta_rule(q, k, v, g, beta, prev, scale):
    """o [T, H, d] of the gated delta rule, each token continuing the state
    of prev[t] (zero state where prev[t] = -1); prev[t] < t."""
    T, H, d = q.shape
    S = np.zeros((T, H, d, d))
    o = np.zeros((T, H, d))
    for t in range(T):
        p = prev[t]
        assert p < t
        for h in range(H):
            a = np.exp(g[t, h])
            Sd = a * S[p, h] if p >= 0 else np.zeros((d, d))
            u = beta[t, h] * (v[t, h] - Sd.T @ k[t, h])
            S[t, h] = Sd + np.outer(k[t, h], u)
            o[t, h] = scale * (S[t, h].T @ q[t, h])
    return o


def gdn_row(plan: Plan, r: int, x, conv_w, g, beta, H: int, d: int, scale: float) -> np.ndarray:
    """Layer core over row r of a packed plan: x [T, 3 H d], conv_w [3 H d, 4],
    g, beta [T, H] -> o [T, H, d] (float64)."""
    prev = path_prev(plan, r)
    y = conv_path(np.asarray(x, np.float64), np.asarray(conv_w, np.float64), prev)
    q, k, v = split_heads(y, H, d)
    return delta_rule(q, k, v, np.asarray(g, np.float64), np.asarray(beta, np.float64), prev, scale)


def gdn_sequence(x, conv_w, g, beta, H: int, d: int, scale: float) -> np.ndarray:
    """The same layer on one unpacked sequence (a plain chain)."""
    L = len(x)
    prev = np.arange(L) - 1
    y = conv_path(np.asarray(x, np.float64), np.asarray(conv_w, np.float64), prev)
    q, k, v = split_heads(y, H, d)
    return delta_rule(q, k, v, np.asarray(g, np.float64), np.asarray(beta, np.float64), prev, scale)
