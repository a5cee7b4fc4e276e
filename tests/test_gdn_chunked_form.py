"""The chunk-wise (WY) algebra of the gated delta rule that the GDN kernels
implement, restated here in float64 and checked against the oracle's
token-by-token recurrence (oracle.gdn.delta_rule) and its reverse mode
(oracle.gdn.delta_rule_grads) on packed trees: segments cut at branch
points, chunks cut from each segment's start (the last one ragged), a child
segment starting from its parent's final state, and, going back, a parent's
end-of-segment state gradient summed over its children.

Per chunk of n tokens, state S0 at its start, gam = cumsum(g) inside it:
  A   = strictly lower (beta_t e^{gam_t - gam_s} k_t . k_s),  T = (I + A)^{-1}
  U^  = T diag(beta) V,   W = T diag(beta e^gam) K,   V' = U^ - W S0
  O   = Q~ S0 + P V'      (Q~ = scale e^gam Q,  P = scale (Q K^T o Gamma))
  S_n = e^{gam_n} S0 + K~^T V'                    (K~ = e^{gam_n - gam} K)
and backwards, from dO and the chunk-end state gradient dS_n:
  dV' = P^T dO + K~ dS_n,   dS0 = Q~^T dO + e^{gam_n} dS_n - W^T dV'
  dQ~ = dO S0^T, dP = dO V'^T, dK~ = V' dS_n^T, dW = -dV' S0^T, dU^ = dV',
  dT  = dU^ (beta V)^T + dW (beta e^gam K)^T,  dA = -strictly lower (T^T dT T^T)
then through the definitions of Q~, K~, P, A, U^, W to q, k, v, beta and gam,
and dg = the reverse cumulative sum of dgam.
"""
import numpy as np
import pytest

from oracle import gdn as OG
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W


def _segments(prev, used):
    """(start, length, parent token) runs: a token continues the previous one's
    segment when it follows it on its path and the previous one has no other child."""
    n_child = np.bincount(prev[:used][prev[:used] >= 0], minlength=used)
    segs = []
    for x in range(used):
        if not (x > 0 and prev[x] == x - 1 and n_child[x - 1] == 1):
            segs.append([x, 0, int(prev[x])])
        segs[-1][1] += 1
    return segs


def _chunk_pieces(Q, K, V, gam, b, S0, scale):
    n = len(gam)
    E = np.exp(gam[:, None] - gam[None, :])
    A = np.tril(b[:, None] * E * (K @ K.T), -1)
    T = np.linalg.inv(np.eye(n) + A)
    BU, BW = b[:, None] * V, (b * np.exp(gam))[:, None] * K
    f = dict(A=A, T=T, BU=BU, BW=BW, Uh=T @ BU, W=T @ BW, Gam=np.tril(E),
             Qt=scale * np.exp(gam)[:, None] * Q, Kt=np.exp(gam[-1] - gam)[:, None] * K)
    f["P"] = scale * (Q @ K.T) * f["Gam"]
    f["Vp"] = f["Uh"] - f["W"] @ S0
    return f


def chunked(prev, used, q, k, v, g, beta, dO, scale, C):
    """(o, dq, dk, dv, dg, dbeta) by the chunk-wise forms, over one row."""
    T, H, d = q.shape
    segs = _segments(prev, used)
    seg_of = np.full(used, -1)
    for i, (s, L, _) in enumerate(segs):
        seg_of[s: s + L] = i
    children = [[] for _ in segs]
    for i, (_, _, p) in enumerate(segs):
        if p >= 0:
            children[seg_of[p]].append(i)
    o = np.zeros((T, H, d))
    grads = [np.zeros((T, H, d)) for _ in range(3)] + [np.zeros((T, H)) for _ in range(2)]
    dq, dk, dv, dg, db = grads
    for h in range(H):
        fin, keep = {}, {}
        for i, (s, L, p) in enumerate(segs):
            S = fin[seg_of[p]].copy() if p >= 0 else np.zeros((d, d))
            for c0 in range(s, s + L, C):
                sl = slice(c0, min(c0 + C, s + L))
                gam, b = np.cumsum(g[sl, h]), beta[sl, h]
                f = _chunk_pieces(q[sl, h], k[sl, h], v[sl, h], gam, b, S, scale)
                o[sl, h] = f["Qt"] @ S + f["P"] @ f["Vp"]
                keep[c0] = (f, S.copy(), gam, b, sl)
                S = np.exp(gam[-1]) * S + f["Kt"].T @ f["Vp"]
            fin[i] = S
        start_grad = {}
        for i in range(len(segs) - 1, -1, -1):     # children come after their parents
            s, L, _ = segs[i]
            dS = sum((start_grad[c] for c in children[i]), np.zeros((d, d)))
            for c0 in reversed(range(s, s + L, C)):
                f, S0, gam, b, sl = keep[c0]
                Q, K, V, dOc = q[sl, h], k[sl, h], v[sl, h], dO[sl, h]
                decay = np.exp(gam[-1])
                dVp = f["P"].T @ dOc + f["Kt"] @ dS
                dS0 = f["Qt"].T @ dOc + decay * dS - f["W"].T @ dVp
                dQt, dP, dKt, dW = dOc @ S0.T, dOc @ f["Vp"].T, f["Vp"] @ dS.T, -dVp @ S0.T
                dgam = (dQt * f["Qt"]).sum(1)
                dQ = scale * np.exp(gam)[:, None] * dQt
                dK = np.exp(gam[-1] - gam)[:, None] * dKt
                kt_term = (dKt * f["Kt"]).sum(1)
                dgam -= kt_term
                dgam[-1] += kt_term.sum() + decay * (dS * S0).sum()
                dPG = dP * f["P"]
                dQ += scale * (dP * f["Gam"]) @ K
                dK += scale * (dP * f["Gam"]).T @ Q
                dgam += dPG.sum(1) - dPG.sum(0)
                dT = dVp @ f["BU"].T + dW @ f["BW"].T
                dBU, dBW = f["T"].T @ dVp, f["T"].T @ dW
                dA = np.tril(-(f["T"].T @ dT @ f["T"].T), -1)
                M = dA * np.tril(np.exp(gam[:, None] - gam[None, :]), -1)   # d/d(beta_t k_t . k_s)
                dK += (M * b[:, None]) @ K + (M * b[:, None]).T @ K
                dbeta_c = (M * (K @ K.T)).sum(1)
                dAA = dA * f["A"]
                dgam += dAA.sum(1) - dAA.sum(0)
                dv[sl, h] += b[:, None] * dBU
                dbeta_c += (dBU * V).sum(1) + np.exp(gam) * (dBW * K).sum(1)
                dK += (b * np.exp(gam))[:, None] * dBW
                dgam += (dBW * f["BW"]).sum(1)
                dg[sl, h] += np.cumsum(dgam[::-1])[::-1]
                db[sl, h] += dbeta_c
                dq[sl, h] += dQ
                dk[sl, h] += dK
                dS = dS0
            start_grad[i] = dS
    return (o, *grads)


@pytest.mark.parametrize("seed,C", [(0, 16), (1, 16), (2, 64), (3, 7)])
def test_chunk_forms_match_the_recurrence(seed, C):
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=1, len_hi=60, row_len=512,
                        min_shared=4, vocab=41)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(seed)
    H, d, scale, T = 2, 6, 0.4, plan.row_len
    used = int(plan.used[0])
    prev = OG.path_prev(plan, 0)[:used]
    q = OG.l2norm(rng.standard_normal((used, H, d)))
    k = OG.l2norm(rng.standard_normal((used, H, d)))
    v = rng.standard_normal((used, H, d))
    g = np.log(rng.uniform(0.7, 1.0, (used, H)))
    beta = rng.uniform(0.1, 0.9, (used, H))
    dO = rng.standard_normal((used, H, d))
    got = chunked(prev, used, q, k, v, g, beta, dO, scale, C)
    want = (OG.delta_rule(q, k, v, g, beta, prev, scale),
            *OG.delta_rule_grads(q, k, v, g, beta, dO, prev, scale))
    for name, a, w in zip(("o", "dq", "dk", "dv", "dg", "dbeta"), got, want):
        np.testing.assert_allclose(a, w, atol=1e-10, err_msg=name)
