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
k_t a fraction beta_t of the way toward v_t).  ``gdn_grads`` is its reverse
mode for L = sum dO . o: a fork's state gradient is the sum over its
children, accumulated as the tokens are visited last to first.

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


# ---------------------------------------------------------------------------
# Backward (reverse mode through the same steps), for the loss
#     L = sum_t sum_h dO[t, h] . o[t, h]
# Tokens are visited in reverse order (a token's children come after it), so
# when token t is reached its state gradient already holds the sum over all
# of its children -- the fork's gradient is the sum of its branches'.
# ---------------------------------------------------------------------------

def _taps(prev: np.ndarray, t: int):
    """(tap, source token) pairs: tap 3 is the token itself, tap 2 one back on
    its path, ... as far as the path goes."""
    out, j = [], t
    for i in range(WIDTH - 1, -1, -1):
        if j < 0:
            break
        out.append((i, j))
        j = prev[j]
    return out


def delta_rule_grads(q, k, v, g, beta, dO, prev, scale):
    """(dq, dk, dv, dg, dbeta) [T, H, ...] of L = sum dO . o for the gated delta
    rule alone (q, k, v given), each token continuing the state of prev[t]."""
    T, H, d = q.shape
    S = np.zeros((T, H, d, d))
    for t in range(T):
        p = prev[t]
        for h in range(H):
            Sp = S[p, h] if p >= 0 else np.zeros((d, d))
            a = np.exp(g[t, h])
            S[t, h] = a * Sp + np.outer(k[t, h], beta[t, h] * (v[t, h] - a * Sp.T @ k[t, h]))

    dS = np.zeros((T, H, d, d))
    dq, dk, dv = np.zeros((T, H, d)), np.zeros((T, H, d)), np.zeros((T, H, d))
    dg, dbeta = np.zeros((T, H)), np.zeros((T, H))
    for t in range(T - 1, -1, -1):
        p = prev[t]
        for h in range(H):
            Sp = S[p, h] if p >= 0 else np.zeros((d, d))
            a, b = np.exp(g[t, h]), beta[t, h]
            dSt = dS[t, h] + scale * np.outer(q[t, h], dO[t, h])
            dq[t, h] = scale * S[t, h] @ dO[t, h]
            w = Sp.T @ k[t, h]                      # the value stored under k before the write
            res = v[t, h] - a * w
            u = b * res
            du = dSt.T @ k[t, h]
            dk[t, h] += dSt @ u
            dv[t, h] += b * du
            dbeta[t, h] = du @ res
            dr = b * du                             # gradient of res
            dk[t, h] += -a * (Sp @ dr)
            dg[t, h] = a * ((dSt * Sp).sum() - w @ dr)
            if p >= 0:
                dS[p, h] += a * dSt - a * np.outer(k[t, h], dr)
    return dq, dk, dv, dg, dbeta


def gdn_grads(x, conv_w, g, beta, dO, prev, H: int, d: int, scale: float):
    """(dx [T, C], dconv_w [C, 4], dg [T, H], dbeta [T, H]) of the layer core
    over one row or sequence whose path predecessors are prev (prev[t] < t)."""
    x = np.asarray(x, np.float64)
    conv_w = np.asarray(conv_w, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    dO = np.asarray(dO, np.float64)
    T, C = x.shape
    z = np.zeros((T, C))
    for t in range(T):
        for i, j in _taps(prev, t):
            z[t] += conv_w[:, i] * x[j]
    sig = 1.0 / (1.0 + np.exp(-z))
    y = z * sig
    raw = [y[:, b * H * d:(b + 1) * H * d].reshape(T, H, d) for b in range(3)]
    nrm = [np.sqrt((raw[b] ** 2).sum(-1, keepdims=True) + EPS) for b in range(2)]
    q, k, v = raw[0] / nrm[0], raw[1] / nrm[1], raw[2]
    dq, dk, dv, dg, dbeta = delta_rule_grads(q, k, v, g, beta, dO, prev, scale)

    dy = np.zeros((T, C))
    for b, dqk in enumerate((dq, dk)):
        qn = (q, k)[b]
        gr = (dqk - qn * (qn * dqk).sum(-1, keepdims=True)) / nrm[b]
        dy[:, b * H * d:(b + 1) * H * d] = gr.reshape(T, H * d)
    dy[:, 2 * H * d:] = dv.reshape(T, H * d)
    dz = dy * sig * (1.0 + z * (1.0 - sig))
    dx, dw = np.zeros((T, C)), np.zeros((C, WIDTH))
    for t in range(T):
        for i, j in _taps(prev, t):
            dx[j] += conv_w[:, i] * dz[t]
            dw[:, i] += x[j] * dz[t]
    return dx, dw, dg, dbeta


def gdn_row_grads(plan: Plan, r: int, x, conv_w, g, beta, dO, H: int, d: int, scale: float):
    """Gradients of the layer core over row r of a packed plan (paths from parent pointers)."""
    return gdn_grads(x, conv_w, g, beta, dO, path_prev(plan, r), H, d, scale)


def gdn_sequence_grads(x, conv_w, g, beta, dO, H: int, d: int, scale: float):
    """The same on one unpacked sequence (a plain chain)."""
    return gdn_grads(x, conv_w, g, beta, dO, np.arange(len(x)) - 1, H, d, scale)
