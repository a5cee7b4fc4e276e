"""Oracle: ancestor sets, tile classes and tree attention (fwd + bwd), float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (prefix-tree-packing page, attention section): a token attends to
its own ancestor chain only -- every ancestor segment fully plus a causal
triangle over its own segment, never a sibling branch or another tree in
the row; most blocks of a packed row are empty and can be skipped.

Ancestors here come from the packer's parent pointers, never from
``subtree_end``; pads (after the last real token of a row) see only
themselves.  For query i of head h (kv head g = h // (Hq/Hkv)) with visible
set V(i):

    s_ij  = scale * q_i . k_j                  (j in V(i))
    LSE_i = ln sum_j exp(s_ij)                 (natural log)
    p_ij  = exp(s_ij - LSE_i),  O_i = sum_j p_ij v_j

and the analytic backward of L = sum_i dO_i . O_i:

    dP_ij = dO_i . v_j,  Delta_i = dO_i . O_i,  dS_ij = p_ij (dP_ij - Delta_i)
    dQ_i  = scale sum_j dS_ij k_j
    dK_j  = scale sum_{i, h in group} dS_ij q_i
    dV_j  = sum_{i, h in group} p_ij dO_i

Tile classes for a (q-tile, k-tile) block: EMPTY when no pair in the block
is visible, FULL when every pair is, PARTIAL otherwise -- counted by brute
force from the visible sets.
"""
from __future__ import annotations

from typing import Dict, List, Tuple

import numpy as np

from .pack import Plan

EMPTY, PARTIAL, FULL = 0, 1, 2


# ---------------------------------------------------------------------------
# Ancestor structure of one packed row
# ---------------------------------------------------------------------------

class RowTree:
    """Visible-key structure of one row, from parent pointers."""

    def __init__(self, plan: Plan, r: int):
        self.T = plan.row_len
        self.used = plan.used[r]
        segs = [rs for rs in plan.row_segments[r] if rs.length > 0]
        by_sid = {rs.sid: rs for rs in plan.row_segments[r]}
        self.segs = segs
        self.seg_of = np.full(self.T, -1, np.int64)
        self.anc: List[List[Tuple[int, int]]] = []   # ancestor row ranges per segment
        for k, rs in enumerate(segs):
            self.seg_of[rs.row_start: rs.row_start + rs.length] = k
            chain = []
            x = rs.parent
            while x >= 0:
                a = by_sid[x]
                if a.length > 0:
                    chain.append((a.row_start, a.row_start + a.length))
                x = a.parent
            self.anc.append(chain[::-1])

    def intervals(self, i: int) -> List[Tuple[int, int]]:
        """Visible keys of query i as disjoint half-open row ranges."""
        k = self.seg_of[i]
        if k < 0:
            return [(i, i + 1)]
        rs = self.segs[k]
        return self.anc[k] + [(rs.row_start, i + 1)]

    def visible(self, i: int) -> np.ndarray:
        return np.concatenate([np.arange(a, b) for a, b in self.intervals(i)])

    def segment_keys(self, k: int):
        """(ancestor key indices, own indices) of segment k."""
        rs = self.segs[k]
        anc = [np.arange(a, b) for a, b in self.anc[k]]
        anc_idx = np.concatenate(anc) if anc else np.zeros(0, np.int64)
        own = np.arange(rs.row_start, rs.row_start + rs.length)
        return anc_idx, own

    def predicate_matrix(self) -> np.ndarray:
        """Boolean [T, T]: entry (i, j) is True iff query i sees key j."""
        M = np.zeros((self.T, self.T), bool)
        for i in range(self.T):
            for a, b in self.intervals(i):
                M[i, a:b] = True
        return M


def useful_pairs(plan: Plan) -> int:
    """Number of visible (query, key) pairs over all real tokens of all rows."""
    tot = 0
    for r in range(plan.n_rows):
        rt = RowTree(plan, r)
        for i in range(rt.used):
            tot += sum(b - a for a, b in rt.intervals(i))
    return tot


def tile_classes(plan: Plan, bm: int = 128, bn: int = 128) -> np.ndarray:
    """int8 [R, T/bm, T/bn] of EMPTY / PARTIAL / FULL, counted from visible sets."""
    T = plan.row_len
    assert T % bm == 0 and T % bn == 0
    out = np.zeros((plan.n_rows, T // bm, T // bn), np.int8)
    for r in range(plan.n_rows):
        rt = RowTree(plan, r)
        ivs = [rt.intervals(i) for i in range(T)]
        depth = max(len(v) for v in ivs)
        LO = np.zeros((T, depth), np.int64)
        HI = np.zeros((T, depth), np.int64)
        for i, v in enumerate(ivs):
            for d, (a, b) in enumerate(v):
                LO[i, d], HI[i, d] = a, b
        for kt in range(T // bn):
            k0, k1 = kt * bn, (kt + 1) * bn
            ov = np.clip(np.minimum(HI, k1) - np.maximum(LO, k0), 0, None).sum(1)
            cnt = ov.reshape(T // bm, bm).sum(1)
            out[r, :, kt] = np.where(cnt == 0, EMPTY, np.where(cnt == bm * bn, FULL, PARTIAL))
    return out


# ---------------------------------------------------------------------------
# Attention, float64
# ---------------------------------------------------------------------------

def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def attn_fwd(plan: Plan, q, k, v, scale: float):
    """O [R,T,Hq,D] and LSE [R,Hq,T] (natural log), float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    R, T, Hq, D = q.shape
    G = Hq // k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((R, Hq, T))
    for r in range(R):
        rt = RowTree(plan, r)
        for kseg in range(len(rt.segs)):
            anc, own = rt.segment_keys(kseg)
            keys = np.concatenate([anc, own])
            mask = np.ones((len(own), len(keys)), bool)
            mask[:, len(anc):] = np.tril(np.ones((len(own), len(own)), bool))
            for h in range(Hq):
                g = h // G
                S = scale * q[r, own, h] @ k[r, keys, g].T
                S = np.where(mask, S, -np.inf)
                m = S.max(1, keepdims=True)
                P = np.exp(S - m)
                l = P.sum(1, keepdims=True)
                lse[r, h, own] = (m + np.log(l))[:, 0]
                o[r, own, h] = (P / l) @ v[r, keys, g]
        pads = np.arange(rt.used, T)
        for h in range(Hq):
            g = h // G
            lse[r, h, pads] = scale * np.einsum("td,td->t", q[r, pads, h], k[r, pads, g])
            o[r, pads, h] = v[r, pads, g]
    return o, lse


def attn_bwd(plan: Plan, q, k, v, do, scale: float):
    """(dQ, dK, dV, O, LSE) for L = sum dO . O, float64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    R, T, Hq, D = q.shape
    G = Hq // k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((R, Hq, T))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r in range(R):
        rt = RowTree(plan, r)
        for kseg in range(len(rt.segs)):
            anc, own = rt.segment_keys(kseg)
            keys = np.concatenate([anc, own])
            mask = np.ones((len(own), len(keys)), bool)
            mask[:, len(anc):] = np.tril(np.ones((len(own), len(own)), bool))
            for h in range(Hq):
                g = h // G
                Kc, Vc, Qs, dOs = k[r, keys, g], v[r, keys, g], q[r, own, h], do[r, own, h]
                S = np.where(mask, scale * Qs @ Kc.T, -np.inf)
                m = S.max(1, keepdims=True)
                P = np.exp(S - m)
                l = P.sum(1, keepdims=True)
                P = P / l
                O = P @ Vc
                o[r, own, h] = O
                lse[r, h, own] = (m + np.log(l))[:, 0]
                dP = dOs @ Vc.T
                delta = (dOs * O).sum(1, keepdims=True)
                dS = P * (dP - delta)
                dq[r, own, h] = scale * dS @ Kc
                dk[r, keys, g] += scale * dS.T @ Qs
                dv[r, keys, g] += P.T @ dOs
        pads = np.arange(rt.used, T)
        for h in range(Hq):
            g = h // G
            # a pad sees only itself: p = 1, O = v, dS = 1 * (dO.v - dO.v) = 0
            lse[r, h, pads] = scale * np.einsum("td,td->t", q[r, pads, h], k[r, pads, g])
            o[r, pads, h] = v[r, pads, g]
            dv[r, pads, g] += do[r, pads, h]
    return dq, dk, dv, o, lse


def query_outputs(rt: RowTree, r: int, i: int, h: int, q, k, v, do, scale: float):
    """O_i, LSE_i and dQ_i of one query (arrays already float64)."""
    G = q.shape[2] // k.shape[2]
    g = h // G
    keys = rt.visible(i)
    s = scale * (k[r, keys, g] @ q[r, i, h])
    m = s.max()
    p = np.exp(s - m)
    l = p.sum()
    p /= l
    O = p @ v[r, keys, g]
    lse = m + np.log(l)
    dP = v[r, keys, g] @ do[r, i, h]
    dS = p * (dP - do[r, i, h] @ O)
    dq = scale * dS @ k[r, keys, g]
    return O, lse, dq


def key_grads(rt: RowTree, r: int, j: int, g: int, q, k, v, do, scale: float):
    """dK_j and dV_j of kv head g, summing every query (and query head of the
    group) whose visible set holds j.  Cost grows with the number of such
    queries, so use it for keys deep in the tree."""
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    dk = np.zeros(k.shape[-1])
    dv = np.zeros(v.shape[-1])
    for i in range(j, rt.T):
        keys = rt.visible(i)
        pos = np.searchsorted(keys, j)
        if pos >= len(keys) or keys[pos] != j:
            continue
        for h in range(g * G, (g + 1) * G):
            s = scale * (k[r, keys, g] @ q[r, i, h])
            m = s.max()
            p = np.exp(s - m)
            p /= p.sum()
            O = p @ v[r, keys, g]
            dP = v[r, keys, g] @ do[r, i, h]
            dS = p * (dP - do[r, i, h] @ O)
            dk += scale * dS[pos] * q[r, i, h]
            dv += p[pos] * do[r, i, h]
    return dk, dv


def queries_seeing(rt: RowTree, j: int) -> int:
    """How many queries of the row see key j."""
    n = 0
    for i in range(j, rt.T):
        if any(a <= j < b for a, b in rt.intervals(i)):
            n += 1
    return n
