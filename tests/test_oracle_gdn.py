"""Pins of the Gated DeltaNet oracle (oracle/gdn.py): closed forms of the
gated delta rule (beta = 0, exact associations under orthonormal keys, a
single key reduces to an unrolled moving average, pure decay), the short
convolution against a library convolution and its tap shifts, and the
packed tree equal to the layer run on every unpacked sequence (state forks,
zero roots, the convolution's hand-off across segments, join copies); its
backward against central finite differences on a packed tree and against
the summed gradients of the unpacked sequences."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import gdn as OG
from oracle import pack as OP
from sft_trie_build_gb300 import workloads as W


def _chain(L):
    return np.arange(L) - 1


def test_beta_zero_keeps_the_state_empty():
    rng = np.random.default_rng(0)
    T, H, d = 9, 2, 4
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    o = OG.delta_rule(q, k, v, -rng.random((T, H)), np.zeros((T, H)), _chain(T), 0.5)
    assert np.all(o == 0.0)


def test_orthonormal_keys_store_exact_associations():
    """No decay, beta = 1, keys e_0, e_1, ...: the state is sum_s k_s v_s^T, so
    querying with k_s returns scale * v_s once s has been written, 0 before."""
    rng = np.random.default_rng(1)
    T, d = 6, 8
    k = np.eye(d)[:T][:, None, :]
    v = rng.standard_normal((T, 1, d))
    for s in range(T):
        q = np.repeat(np.eye(d)[s][None, None, :], T, 0)
        o = OG.delta_rule(q, k, v, np.zeros((T, 1)), np.ones((T, 1)), _chain(T), 0.25)
        for t in range(T):
            want = 0.25 * v[s, 0] if t >= s else np.zeros(d)
            np.testing.assert_allclose(o[t, 0], want, atol=1e-12)


def test_single_key_is_an_unrolled_moving_average():
    """One unit key for every token: the value read back under it is
    r_t = sum_{s<=t} beta_s v_s prod_{s<u<=t} (1 - beta_u) alpha_u, a
    closed form that keeps alpha inside the correction term."""
    rng = np.random.default_rng(2)
    T, d = 12, 5
    key = rng.standard_normal(d)
    key /= np.linalg.norm(key)
    k = np.tile(key, (T, 1))[:, None, :]
    v = rng.standard_normal((T, 1, d))
    g = np.log(rng.uniform(0.5, 1.0, (T, 1)))
    beta = rng.uniform(0.05, 0.95, (T, 1))
    o = OG.delta_rule(k.copy(), k, v, g, beta, _chain(T), 1.0)
    a = np.exp(g[:, 0])
    for t in range(T):
        want = np.zeros(d)
        for s in range(t + 1):
            w = beta[s, 0] * np.prod([(1 - beta[u, 0]) * a[u] for u in range(s + 1, t + 1)])
            want += w * v[s, 0]
        np.testing.assert_allclose(o[t, 0], want, atol=1e-12)


def test_pure_decay():
    """beta_1 = 1, then 0: the stored value decays by exp(sum g) and nothing else."""
    rng = np.random.default_rng(3)
    T, d = 7, 4
    key = np.eye(d)[2]
    k = np.tile(key, (T, 1))[:, None, :]
    v = rng.standard_normal((T, 1, d))
    g = -rng.random((T, 1))
    beta = np.zeros((T, 1))
    beta[0] = 1.0
    o = OG.delta_rule(k.copy(), k, v, g, beta, _chain(T), 1.0)
    for t in range(T):
        np.testing.assert_allclose(o[t, 0], np.exp(g[1:t + 1, 0].sum()) * v[0, 0], atol=1e-12)


def test_conv_taps_and_library_convolution():
    rng = np.random.default_rng(4)
    L, C = 10, 6
    x = rng.standard_normal((L, C))
    silu = lambda z: z * expit(z)  # noqa: E731
    w = np.zeros((C, 4))
    w[:, 3] = 1.0
    np.testing.assert_allclose(OG.conv_path(x, w, _chain(L)), silu(x), atol=1e-12)
    w = np.zeros((C, 4))
    w[:, 0] = 1.0
    shifted = np.vstack([np.zeros((3, C)), x[:-3]])
    np.testing.assert_allclose(OG.conv_path(x, w, _chain(L)), silu(shifted), atol=1e-12)
    w = rng.standard_normal((C, 4))
    want = np.stack([np.convolve(x[:, c], w[c, ::-1])[:L] for c in range(C)], 1)
    np.testing.assert_allclose(OG.conv_path(x, w, _chain(L)), silu(want), atol=1e-12)


def test_l2norm_gives_unit_heads():
    rng = np.random.default_rng(5)
    y = rng.standard_normal((5, 3 * 2 * 4)) * 3
    q, k, _ = OG.split_heads(y, 2, 4)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, atol=1e-6)
    np.testing.assert_allclose(np.linalg.norm(k, axis=-1), 1.0, atol=1e-6)


def _token_inputs(rng, V, P, H, d):
    """Per-(token, position) inputs, so a sequence's inputs do not depend on the packing."""
    C = 3 * H * d
    Ex, Px = rng.standard_normal((V, C)), 0.5 * rng.standard_normal((P, C))
    Eg, Eb = np.log(rng.uniform(0.8, 1.0, (V, H))), rng.uniform(0.1, 0.9, (V, H))
    Pg = np.log(rng.uniform(0.9, 1.0, (P, H)))
    return (lambda t, p: Ex[t] + Px[p]), (lambda t, p: Eg[t] + Pg[p]), (lambda t, p: Eb[t])


@pytest.mark.parametrize("seed", range(4))
def test_packed_tree_equals_unpacked_sequences(seed):
    b = W.random_forest(seed, n_roots=3, max_depth=3, max_children=3, len_lo=3, len_hi=30, row_len=256,
                        min_shared=4, vocab=53)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(seed)
    H, d, scale = 2, 4, 0.5
    fx, fg, fb = _token_inputs(rng, 53, b.row_len, H, d)
    conv_w = 0.5 * rng.standard_normal((3 * H * d, 4))
    outs = []
    for r in range(plan.n_rows):
        tok, pos = plan.token_ids[r], plan.position_ids[r]
        x = np.stack([fx(t, p) for t, p in zip(tok, pos)])
        g = np.stack([fg(t, p) for t, p in zip(tok, pos)])
        beta = np.stack([fb(t, p) for t, p in zip(tok, pos)])
        outs.append(OG.gdn_row(plan, r, x, conv_w, g, beta, H, d, scale))
    o = np.concatenate(outs)          # [R * T, H, d]
    offs = np.concatenate([[0], np.cumsum([len(s) for s in b.seqs])])
    for s, seq in enumerate(b.seqs):
        x = np.stack([fx(t, p) for p, t in enumerate(seq)])
        g = np.stack([fg(t, p) for p, t in enumerate(seq)])
        beta = np.stack([fb(t, p) for p, t in enumerate(seq)])
        want = OG.gdn_sequence(x, conv_w, g, beta, H, d, scale)
        got = o[plan.gather_index[offs[s]: offs[s + 1]]]
        np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-10)


def test_pads_are_their_own_roots():
    b = W.random_forest(9, n_roots=2, max_depth=2, len_lo=3, len_hi=20, row_len=256, min_shared=4, vocab=31)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    used = int(plan.used[0])
    assert used < plan.row_len
    prev = OG.path_prev(plan, 0)
    assert np.all(prev[used:] == -1)
    assert np.all(prev[:used] < np.arange(used))


def _fd_check(x, w, g, b, dO, prev, H, d, scale, rng, n=6):
    grads = OG.gdn_grads(x, w, g, b, dO, prev, H, d, scale)

    def loss(args):
        y = OG.conv_path(args[0], args[1], prev)
        q, k, v = OG.split_heads(y, H, d)
        return (OG.delta_rule(q, k, v, args[2], args[3], prev, scale) * dO).sum()

    base = [x, w, g, b]
    eps = 1e-6
    for a_i, grad in enumerate(grads):
        for _ in range(n):
            idx = tuple(int(rng.integers(0, s)) for s in base[a_i].shape)
            plus = [t.copy() for t in base]
            minus = [t.copy() for t in base]
            plus[a_i][idx] += eps
            minus[a_i][idx] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * (1 + abs(fd)), (a_i, idx, fd, grad[idx])


def test_backward_matches_finite_differences_on_a_tree():
    """Central differences in float64 on a packed row with forks and pads:
    every input (x, the convolution weights, g, beta)."""
    b = W.random_forest(5, n_roots=2, max_depth=2, max_children=3, len_lo=2, len_hi=8, row_len=64,
                        min_shared=2, vocab=17)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(6)
    H, d, T = 2, 3, plan.row_len
    x = rng.standard_normal((T, 3 * H * d))
    w = 0.5 * rng.standard_normal((3 * H * d, 4))
    g = np.log(rng.uniform(0.6, 1.0, (T, H)))
    beta = rng.uniform(0.1, 0.9, (T, H))
    dO = rng.standard_normal((T, H, d))
    _fd_check(x, w, g, beta, dO, OG.path_prev(plan, 0), H, d, 0.7, rng)


@pytest.mark.parametrize("seed", range(3))
def test_backward_packed_equals_sum_over_unpacked(seed):
    """With dO split evenly over the copies of a shared position, the packed
    gradients equal the sum of the unpacked sequences' gradients: per input
    token over its copies, and for the weights over all sequences (a
    branch point's state gradient is the sum over its branches)."""
    b = W.random_forest(seed, n_roots=2, max_depth=3, max_children=3, len_lo=2, len_hi=25, row_len=256,
                        min_shared=3, vocab=29)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    rng = np.random.default_rng(seed)
    H, d, scale = 2, 3, 0.5
    R, T = plan.n_rows, plan.row_len
    x = rng.standard_normal((R * T, 3 * H * d))
    w = 0.5 * rng.standard_normal((3 * H * d, 4))
    g = np.log(rng.uniform(0.7, 1.0, (R * T, H)))
    beta = rng.uniform(0.1, 0.9, (R * T, H))
    dO = rng.standard_normal((R * T, H, d))
    mult = np.bincount(plan.gather_index, minlength=R * T).astype(np.float64)
    dO_packed = np.where(mult[:, None, None] > 0, dO, 0.0)
    want_x, want_g, want_b = np.zeros_like(x), np.zeros_like(g), np.zeros_like(beta)
    want_w = np.zeros_like(w)
    offs = np.concatenate([[0], np.cumsum([len(s) for s in b.seqs])])
    for s in range(len(b.seqs)):
        idx = plan.gather_index[offs[s]: offs[s + 1]]
        gx, gw, gg, gb = OG.gdn_sequence_grads(x[idx], w, g[idx], beta[idx],
                                                dO[idx] / mult[idx][:, None, None], H, d, scale)
        np.add.at(want_x, idx, gx)
        np.add.at(want_g, idx, gg)
        np.add.at(want_b, idx, gb)
        want_w += gw
    got_w = np.zeros_like(w)
    for r in range(R):
        sl = slice(r * T, (r + 1) * T)
        gx, gw, gg, gb = OG.gdn_row_grads(plan, r, x[sl], w, g[sl], beta[sl], dO_packed[sl], H, d, scale)
        np.testing.assert_allclose(gx, want_x[sl], atol=1e-10)
        np.testing.assert_allclose(gg, want_g[sl], atol=1e-10)
        np.testing.assert_allclose(gb, want_b[sl], atol=1e-10)
        got_w += gw
    np.testing.assert_allclose(got_w, want_w, atol=1e-9)


def test_backward_per_head_slices_equal_the_full_layer():
    """Heads never mix: the layer on one head's channels (H = 1) gives that
    head's slice of the full layer's gradients (what the full-size GPU test
    compares against)."""
    import sys
    import os
    import torch
    sys.path.insert(0, os.path.dirname(__file__))
    from gdn_helpers import oracle_head_grads, oracle_row_grads

    b = W.random_forest(4, n_roots=2, max_depth=2, max_children=3, len_lo=2, len_hi=12, row_len=64,
                        min_shared=2, vocab=17)
    plan = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared)
    H, d = 3, 128
    gen = torch.Generator().manual_seed(3)
    N = plan.n_rows * plan.row_len
    x = torch.randn(N, 3 * H * d, generator=gen).to(torch.bfloat16)
    cw = torch.randn(3 * H * d, 4, generator=gen) * 0.5
    g = torch.log(0.85 + 0.15 * torch.rand(N, H, generator=gen))
    beta = torch.sigmoid(torch.randn(N, H, generator=gen))
    dO = np.random.default_rng(3).standard_normal((N, H, d))
    full = oracle_row_grads(plan, H, (x, cw, g, beta), dO, 0.1)
    T = plan.row_len
    assert plan.n_rows > 1
    wsum = {0: 0.0, 2: 0.0}
    for r in range(plan.n_rows):
        sl = slice(r * T, (r + 1) * T)
        for h, (ch, gx, gw, gg, gb) in oracle_head_grads(plan, r, (x, cw, g, beta), dO, 0.1, H, (0, 2)).items():
            np.testing.assert_allclose(gx, full[0][sl][:, ch], atol=1e-12)
            np.testing.assert_allclose(gg, full[2][sl, h], atol=1e-12)
            np.testing.assert_allclose(gb, full[3][sl, h], atol=1e-12)
            wsum[h] = wsum[h] + gw
    for h in (0, 2):
        ch = np.concatenate([np.arange(bb * H * 128 + h * 128, bb * H * 128 + (h + 1) * 128) for bb in range(3)])
        np.testing.assert_allclose(wsum[h], full[1][ch], atol=1e-12)
