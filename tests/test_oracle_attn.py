"""Pins of the attention oracle: a library causal attention, the unpacked
equivalence the pages claim (packing leaves every sequence's outputs and
gradients unchanged), finite differences, and brute-force tile classes."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attn as A
from oracle import pack as P
from sft_trie_build_gb300 import workloads as W


def _tensors(R, T, Hq, Hkv, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(R, T, Hq, D, generator=g, dtype=torch.float64) * std
    k = torch.randn(R, T, Hkv, D, generator=g, dtype=torch.float64) * std
    v = torch.randn(R, T, Hkv, D, generator=g, dtype=torch.float64) * std
    do = torch.randn(R, T, Hq, D, generator=g, dtype=torch.float64)
    return q, k, v, do


def _small_plan(seed, row_len=256, min_shared=4):
    b = W.random_forest(seed, n_roots=2, max_depth=3, len_lo=2, len_hi=24,
                        row_len=row_len, min_shared=min_shared)
    return b, P.pack(b.seqs, b.trainable, row_len, min_shared, b.family)


def test_single_chain_is_causal_attention():
    T, D, H = 96, 32, 2
    seqs = [np.arange(T, dtype=np.int32)]
    plan = P.pack(seqs, [np.zeros(T, np.uint8)], T, 64)
    q, k, v, _ = _tensors(1, T, H, H, D, 0)
    scale = D ** -0.5
    o, lse = A.attn_fwd(plan, q, k, v, scale)
    ref = F.scaled_dot_product_attention(q[0].transpose(0, 1), k[0].transpose(0, 1),
                                         v[0].transpose(0, 1), is_causal=True, scale=scale)
    np.testing.assert_allclose(o[0], ref.transpose(0, 1).numpy(), atol=1e-12)
    # LSE normalizes the causal softmax: exp(S - LSE) @ V reproduces SDPA
    S = scale * torch.einsum("thd,shd->hts", q[0], k[0]).numpy()
    causal = np.tril(np.ones((T, T), bool))
    Pm = np.where(causal, np.exp(S - lse[0][:, :, None]), 0.0)
    O2 = np.einsum("hts,shd->thd", Pm, v[0].numpy())
    np.testing.assert_allclose(O2, ref.transpose(0, 1).numpy(), atol=1e-12)


def _unpacked_reference(plan, b, q, k, v, do, scale):
    """Per-sequence causal attention (torch SDPA) on the unpacked sequences,
    differentiated by autograd.  A packed token shared by m sequences appears
    m times unpacked; each copy of its query gets dO / m, so the unpacked loss
    equals the packed one and autograd sums gradients over the copies."""
    T = plan.row_len
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    qf = q.reshape(-1, Hq, q.shape[-1]).clone().requires_grad_(True)
    kf = k.reshape(-1, Hkv, k.shape[-1]).clone().requires_grad_(True)
    vf = v.reshape(-1, Hkv, v.shape[-1]).clone().requires_grad_(True)
    dof = do.reshape(-1, Hq, do.shape[-1])
    offs = np.concatenate([[0], np.cumsum([len(s) for s in b.seqs])])
    mult = np.bincount(plan.gather_index, minlength=plan.n_rows * T)
    loss = 0
    outs = []
    for s in range(len(b.seqs)):
        gi = torch.from_numpy(plan.gather_index[offs[s]:offs[s + 1]])
        qs = qf[gi].transpose(0, 1)                       # [Hq, L, D]
        ks = kf[gi].repeat_interleave(G, dim=1).transpose(0, 1)
        vs = vf[gi].repeat_interleave(G, dim=1).transpose(0, 1)
        o = F.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=scale)
        w = dof[gi].transpose(0, 1) / torch.from_numpy(mult[gi.numpy()]).to(o.dtype)[None, :, None]
        loss = loss + (o * w).sum()
        outs.append((gi, o.detach().transpose(0, 1)))
    loss.backward()
    return outs, qf.grad.reshape(q.shape), kf.grad.reshape(k.shape), vf.grad.reshape(v.shape)


@pytest.mark.parametrize("seed", range(6))
def test_unpacked_equivalence(seed):
    b, plan = _small_plan(seed)
    R, T = plan.n_rows, plan.row_len
    Hq, Hkv, D = 4, 2, 16
    q, k, v, do = _tensors(R, T, Hq, Hkv, D, seed)
    scale = D ** -0.5
    dq, dk, dv, o, lse = A.attn_bwd(plan, q, k, v, do, scale)
    o2, lse2 = A.attn_fwd(plan, q, k, v, scale)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)
    outs, rq, rk, rv = _unpacked_reference(plan, b, q, k, v, do, scale)
    of = o.reshape(-1, Hq, D)
    for gi, ref in outs:
        np.testing.assert_allclose(of[gi.numpy()], ref.numpy(), atol=1e-10)
    # gradients at every real token (pads are outside every sequence)
    real = np.zeros((R, T), bool)
    for r in range(R):
        real[r, :plan.used[r]] = True
    np.testing.assert_allclose(dq[real], rq.numpy()[real], atol=1e-10)
    np.testing.assert_allclose(dk[real], rk.numpy()[real], atol=1e-10)
    np.testing.assert_allclose(dv[real], rv.numpy()[real], atol=1e-10)


def test_pads_see_only_themselves():
    b, plan = _small_plan(3, row_len=384)
    R, T = plan.n_rows, plan.row_len
    q, k, v, do = _tensors(R, T, 2, 1, 8, 1)
    dq, dk, dv, o, lse = A.attn_bwd(plan, q, k, v, do, 0.3)
    for r in range(R):
        u = plan.used[r]
        assert u < T
        np.testing.assert_allclose(o[r, u:, 0], v.numpy()[r, u:, 0])
        np.testing.assert_allclose(lse[r, 0, u:], 0.3 * (q[r, u:, 0] * k[r, u:, 0]).sum(-1).numpy())
        assert np.abs(dq[r, u:]).max() == 0 and np.abs(dk[r, u:]).max() == 0
        np.testing.assert_allclose(dv[r, u:, 0], do.numpy()[r, u:, 0] + do.numpy()[r, u:, 1])


def test_finite_differences():
    """Central differences of L = sum dO . O in float64 on a tiny tree."""
    b = W.tiny(0)
    plan = P.pack(b.seqs, b.trainable, b.row_len, 64)
    T, D = plan.row_len, 8
    q, k, v, do = _tensors(1, T, 2, 1, D, 7)
    scale = 0.35
    dq, dk, dv, _, _ = A.attn_bwd(plan, q, k, v, do, scale)
    dn = do.numpy()

    def loss(qq, kk, vv):
        o, _ = A.attn_fwd(plan, qq, kk, vv, scale)
        return float((o * dn).sum())

    rng = np.random.default_rng(0)
    eps = 1e-6
    qn, kn, vn = q.numpy().copy(), k.numpy().copy(), v.numpy().copy()
    u = plan.used[0]
    for name, arr, grad in (("q", qn, dq), ("k", kn, dk), ("v", vn, dv)):
        for _ in range(4):
            idx = (0, int(rng.integers(0, u)), int(rng.integers(0, arr.shape[2])), int(rng.integers(0, D)))
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss(qn, kn, vn)
            arr[idx] = old - eps
            lm = loss(qn, kn, vn)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("seed", range(5))
def test_tile_classes_brute_force(seed):
    b, plan = _small_plan(seed, row_len=512, min_shared=4)
    for bm in (64, 128):
        cls = A.tile_classes(plan, bm, bm)
        for r in range(plan.n_rows):
            M = A.RowTree(plan, r).predicate_matrix()
            nt = plan.row_len // bm
            blocks = M.reshape(nt, bm, nt, bm).transpose(0, 2, 1, 3)
            want = np.where(~blocks.any((2, 3)), A.EMPTY,
                            np.where(blocks.all((2, 3)), A.FULL, A.PARTIAL))
            assert (cls[r] == want).all()
            # the subtree_end interval predicate gives the same matrix
            se = plan.subtree_end[r]
            j = np.arange(plan.row_len)
            Mse = (j[None, :] <= j[:, None]) & (se[None, :] >= j[:, None])
            assert (Mse == M).all()
            # upper-triangle tiles are empty, diagonal tiles partial
            iu = np.triu_indices(nt, 1)
            assert (cls[r][iu] == A.EMPTY).all()
            assert (np.diag(cls[r]) == A.PARTIAL).all()


def test_sampled_functions_match_full():
    b, plan = _small_plan(11, row_len=256)
    R, T = plan.n_rows, plan.row_len
    q, k, v, do = (x.numpy() for x in _tensors(R, T, 4, 2, 16, 5))
    scale = 0.25
    dq, dk, dv, o, lse = A.attn_bwd(plan, q, k, v, do, scale)
    rng = np.random.default_rng(1)
    for r in range(R):
        rt = A.RowTree(plan, r)
        for i in rng.integers(0, T, 8):
            for h in range(4):
                oi, li, dqi = A.query_outputs(rt, r, int(i), h, q, k, v, do, scale)
                np.testing.assert_allclose(oi, o[r, i, h], atol=1e-12)
                np.testing.assert_allclose(li, lse[r, h, i], atol=1e-12)
                np.testing.assert_allclose(dqi, dq[r, i, h], atol=1e-12)
        for j in rng.integers(0, plan.used[r], 4):
            for g in range(2):
                dkj, dvj = A.key_grads(rt, r, int(j), g, q, k, v, do, scale)
                np.testing.assert_allclose(dkj, dk[r, j, g], atol=1e-12)
                np.testing.assert_allclose(dvj, dv[r, j, g], atol=1e-12)


def test_gradient_sum_identities():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per kv group (softmax rows
    sum to one); used at full sizes where only samples are affordable."""
    b, plan = _small_plan(2, row_len=256)
    q, k, v, do = (x.numpy() for x in _tensors(plan.n_rows, plan.row_len, 4, 2, 16, 9))
    dq, dk, dv, _, _ = A.attn_bwd(plan, q, k, v, do, 0.25)
    np.testing.assert_allclose(dk.sum(1), 0, atol=1e-10)
    dsum = do.reshape(do.shape[0], do.shape[1], 2, 2, -1).sum(3).sum(1)
    np.testing.assert_allclose(dv.sum(1), dsum, atol=1e-10)
