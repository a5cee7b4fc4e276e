"""GPU path vs the oracle, through the C ABI.

* tile classes: bit-exact;
* float32: max abs <= 1e-5;
* bf16: O <= 1e-2 and LSE <= 1e-3 max abs; dQ/dK/dV max|diff| / max|ref| <= 2e-2,
  against the oracle run on the same bf16-rounded inputs upcast to float64.
Small cases compare every element; the workload-sized cases compare sampled
queries (O, LSE, dQ), sampled keys deep in the tree (dK, dV), and the sum
identities sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per kv head.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, FP32_TOL, GpuRun, pack_both, rel_err
from oracle import attn as OA
from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(stp_lib):
    return stp_lib


def _small_batch(seed, row_len, n_roots=3, len_hi=120, ms=16):
    return W.random_forest(seed, n_roots=n_roots, max_depth=3, max_children=3, len_lo=8,
                           len_hi=len_hi, row_len=row_len, min_shared=ms, vocab=W.VOCAB)


# --- tile classification ---------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "grpo", "curriculum", "deep", "bushy"])
def test_tile_classes_workloads(name):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    R, T = se.shape
    g = GpuRun(se, 1, 1, 64, stp.STP_FP32, 0.125,
               torch.zeros(R, T, 1, 64), torch.zeros(R, T, 1, 64), torch.zeros(R, T, 1, 64))
    g.classify()
    np.testing.assert_array_equal(g.tile_classes(), OA.tile_classes(ref))
    assert stp.stp_device_status(g.buf.tile_meta) == stp.STP_OK


@pytest.mark.parametrize("seed", range(6))
def test_tile_classes_random(seed):
    b = _small_batch(seed, 1024 + 128 * (seed % 3))
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    R, T = se.shape
    z = torch.zeros(R, T, 1, 64)
    g = GpuRun(se, 1, 1, 64, stp.STP_FP32, 0.125, z, z, z)
    g.classify()
    np.testing.assert_array_equal(g.tile_classes(), OA.tile_classes(ref))


def test_classify_flags_bad_subtree_end():
    T = 256
    se = np.arange(T, dtype=np.int32)[None].copy()
    se[0, 10] = 5          # exit index before the token itself
    z = torch.zeros(1, T, 1, 64)
    g = GpuRun(se, 1, 1, 64, stp.STP_FP32, 0.125, z, z, z)
    g.classify()
    assert stp.stp_device_status(g.buf.tile_meta) == stp.STP_EDEVICE


# --- float32 ----------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 5, 9])
def test_fp32_tiny_forward(seed):
    b = W.tiny(seed)
    out, info, ref = pack_both(b)
    shape = W.attn_shape("tiny", info["n_rows"], b.row_len)
    q, k, v, do = W.attn_tensors(shape, seed)
    g = GpuRun(out["subtree_end"], 1, 1, 64, stp.STP_FP32, shape.scale, q, k, v, do).run(backward=False)
    o_ref, lse_ref = OA.attn_fwd(ref, q, k, v, shape.scale)
    assert np.abs(g.o.cpu().numpy() - o_ref).max() <= FP32_TOL
    assert np.abs(g.lse.cpu().numpy() - lse_ref).max() <= FP32_TOL


@pytest.mark.parametrize("D", [64, 128])
def test_fp32_forward_backward_small(D):
    b = _small_batch(3, 512)
    out, info, ref = pack_both(b)
    shape = W.AttnShape(info["n_rows"], 512, 4, 2, D, "fp32", D ** -0.5, 1.0)
    q, k, v, do = W.attn_tensors(shape, 3)
    g = GpuRun(out["subtree_end"], 4, 2, D, stp.STP_FP32, shape.scale, q, k, v, do).run()
    dq, dk, dv, o, lse = OA.attn_bwd(ref, q, k, v, do, shape.scale)
    assert np.abs(g.o.cpu().numpy() - o).max() <= FP32_TOL
    assert np.abs(g.lse.cpu().numpy() - lse).max() <= FP32_TOL
    for got, want in ((g.dq, dq), (g.dk, dk), (g.dv, dv)):
        assert np.abs(got.cpu().numpy() - want).max() <= 1e-4


# --- bf16, every element ---------------------------------------------------

@pytest.mark.parametrize("heads", [(4, 2), (8, 2), (2, 2), (3, 1)])
@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_small_every_element(heads, seed):
    Hq, Hkv = heads
    b = _small_batch(10 + seed, 1024, n_roots=4, len_hi=160, ms=16)
    out, info, ref = pack_both(b)
    R = info["n_rows"]
    shape = W.AttnShape(R, 1024, Hq, Hkv, 128, "bf16", 128 ** -0.5, 0.5)
    q, k, v, do = W.attn_tensors(shape, seed)
    g = GpuRun(out["subtree_end"], Hq, Hkv, 128, stp.STP_BF16, shape.scale, q, k, v, do).run()
    dq, dk, dv, o, lse = OA.attn_bwd(ref, q, k, v, do, shape.scale)
    assert np.abs(g.o.float().cpu().numpy() - o).max() <= BF16_TOL["o"]
    assert np.abs(g.lse.cpu().numpy() - lse).max() <= BF16_TOL["lse"]
    assert rel_err(g.dq.float().cpu().numpy(), dq) <= BF16_TOL["grad_rel"]
    assert rel_err(g.dk.float().cpu().numpy(), dk) <= BF16_TOL["grad_rel"]
    assert rel_err(g.dv.float().cpu().numpy(), dv) <= BF16_TOL["grad_rel"]


def test_bf16_single_tile_row_and_all_pads():
    """One 128-token row with a 5-token sequence: one diagonal tile, mostly pads."""
    seqs = [np.arange(5, dtype=np.int32)]
    b = W.SeqBatch(seqs, [np.array([0, 0, 1, 1, 1], np.uint8)], None, 128, 64)
    out, info, ref = pack_both(b)
    shape = W.AttnShape(1, 128, 2, 1, 128, "bf16", 128 ** -0.5, 0.5)
    q, k, v, do = W.attn_tensors(shape, 4)
    g = GpuRun(out["subtree_end"], 2, 1, 128, stp.STP_BF16, shape.scale, q, k, v, do).run()
    dq, dk, dv, o, lse = OA.attn_bwd(ref, q, k, v, do, shape.scale)
    assert np.abs(g.o.float().cpu().numpy() - o).max() <= BF16_TOL["o"]
    assert np.abs(g.lse.cpu().numpy() - lse).max() <= BF16_TOL["lse"]
    assert rel_err(g.dv.float().cpu().numpy(), dv) <= BF16_TOL["grad_rel"]


def test_empty_descriptor_is_noop():
    d = stp.Desc(0, 256, 2, 1, 128, stp.STP_BF16)
    buf = stp.Buffers(d)
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    se = torch.empty(4, dtype=torch.int32, device="cuda")
    stp.stp_classify(d, se, buf.tile_meta)
    stp.stp_attn_fwd(d, x, x, x, se, buf.tile_meta, x, x.float(), buf.fwd_ws)


def test_bwd_capacity_too_small_is_flagged():
    """A dS workspace one pair short: classification and the backward report a
    device error instead of writing past the workspace."""
    b = _small_batch(2, 1024)
    out, info, ref = pack_both(b)
    se = out["subtree_end"]
    R, T = se.shape
    need = stp.stp_count_tile_pairs(se)
    assert need == int((OA.tile_classes(ref) != OA.EMPTY).sum())
    shape = W.AttnShape(R, T, 4, 2, 128, "bf16", 128 ** -0.5, 0.5)
    q, k, v, do = W.attn_tensors(shape, 1)
    g = GpuRun(se, 4, 2, 128, stp.STP_BF16, shape.scale, q, k, v, do)
    g.desc = stp.Desc(R, T, 4, 2, 128, stp.STP_BF16, shape.scale, need - 1)
    g.buf = stp.Buffers(g.desc)
    g.classify()
    g.fwd()
    g.bwd()
    torch.cuda.synchronize()
    assert stp.stp_device_status(g.buf.tile_meta) == stp.STP_EDEVICE
    assert stp.stp_device_status(g.buf.bwd_ws) == stp.STP_EDEVICE


def test_misaligned_pointer_rejected():
    d = stp.Desc(1, 256, 2, 1, 128, stp.STP_BF16)
    buf = stp.Buffers(d)
    x = torch.zeros(1 * 256 * 2 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    se = torch.arange(256, dtype=torch.int32, device="cuda")
    lse = torch.empty(2 * 256, dtype=torch.float32, device="cuda")
    stp.stp_classify(d, se, buf.tile_meta)
    with pytest.raises(stp.StpError) as e:
        stp.stp_attn_fwd(d, x[1:].data_ptr(), x, x, se, buf.tile_meta, x, lse, buf.fwd_ws)
    assert e.value.status == stp.STP_EINVAL


# --- workload sizes, sampled ---------------------------------------------

def _sample_checks(name, n_queries=24, n_keys=6, seed=0):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    _sample_checks_batch(b, lambda R, T: W.attn_shape(name, R, T), n_queries, n_keys, seed)


def _sample_checks_batch(b, shape_of, n_queries=24, n_keys=6, seed=0):
    out, info, ref = pack_both(b)
    R, T = info["n_rows"], b.row_len
    shape = shape_of(R, T)
    q, k, v, do = W.attn_tensors(shape, seed)
    g = GpuRun(out["subtree_end"], shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
               stp.STP_BF16, shape.scale, q, k, v, do).run()
    qn, kn, vn, dn = (x.double().numpy() for x in (q, k, v, do))
    o_g = g.o.float().cpu().numpy()
    lse_g = g.lse.cpu().numpy()
    dq_g = g.dq.float().cpu().numpy()
    dk_g = g.dk.float().cpu().numpy()
    dv_g = g.dv.float().cpu().numpy()
    rng = np.random.default_rng(seed)
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    errs = {"o": 0.0, "lse": 0.0}
    dq_pairs, dk_pairs, dv_pairs = [], [], []
    for _ in range(n_queries):
        r = int(rng.integers(0, R))
        rt = OA.RowTree(ref, r)
        i = int(rng.integers(0, T))
        h = int(rng.integers(0, Hq))
        o_i, lse_i, dq_i = OA.query_outputs(rt, r, i, h, qn, kn, vn, dn, shape.scale)
        errs["o"] = max(errs["o"], np.abs(o_g[r, i, h] - o_i).max())
        errs["lse"] = max(errs["lse"], abs(lse_g[r, h, i] - lse_i))
        dq_pairs.append((dq_g[r, i, h], dq_i))
    # keys whose queries are few: the last tokens of leaf segments
    for _ in range(n_keys):
        r = int(rng.integers(0, R))
        rt = OA.RowTree(ref, r)
        leaves = [s for s in ref.row_segments[r] if s.length > 0 and
                  ref.trie.segments[s.sid].is_leaf]
        s = leaves[int(rng.integers(0, len(leaves)))]
        j = s.row_start + s.length - 1 - int(rng.integers(0, min(s.length, 40)))
        gg = int(rng.integers(0, Hkv))
        dk_j, dv_j = OA.key_grads(rt, r, j, gg, qn, kn, vn, dn, shape.scale)
        dk_pairs.append((dk_g[r, j, gg], dk_j))
        dv_pairs.append((dv_g[r, j, gg], dv_j))
    assert errs["o"] <= BF16_TOL["o"], errs
    assert errs["lse"] <= BF16_TOL["lse"], errs
    for pairs in (dq_pairs, dk_pairs, dv_pairs):
        got = np.stack([p[0] for p in pairs])
        want = np.stack([p[1] for p in pairs])
        assert rel_err(got, want) <= BF16_TOL["grad_rel"]
    # identities over every key: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i (per kv head)
    G = Hq // Hkv
    dsum = dn.reshape(R, T, Hkv, G, -1).sum(3).sum(1)
    scale_dv = np.abs(dv_g).max() * np.sqrt(T)
    assert np.abs(dv_g.astype(np.float64).sum(1) - dsum).max() <= 2e-2 * scale_dv
    assert np.abs(dk_g.astype(np.float64).sum(1)).max() <= 2e-2 * np.abs(dk_g).max() * np.sqrt(T)


@pytest.mark.parametrize("name", ["grpo", "curriculum", "deep", "bushy"])
def test_bf16_workload_sampled(name):
    _sample_checks(name)


def test_bf16_longest_rows_sampled():
    """The longest rows the library accepts: the prefix-tree-packing page's
    32-rollout batch packed into two rows of 131072 tokens (130,105 and
    122,114 used; lists of up to ~220 key tiles), two query heads on one kv
    head, bf16: classification, forward and backward in one launch each;
    sampled queries (O, LSE, dQ) and keys near leaf ends (dK, dV) against
    the oracle, and the sum identities over every key."""
    b = W.rollout32(0)
    _sample_checks_batch(b, lambda R, T: W.AttnShape(R, T, 2, 1, 128, "bf16", 128 ** -0.5, 0.5),
                         n_queries=16, n_keys=6, seed=3)


# --- bounded dS workspace ----------------------------------------------------

@pytest.mark.parametrize("name,heads,ds_groups", [("small", (8, 4), (1, 3)), ("grpo", None, (2,))])
def test_bwd_ds_groups_bit_identical(name, heads, ds_groups):
    """Holding the dS tiles of fewer kv-head groups at once (a smaller
    workspace; groups then wait for the slot's previous user) gives the same
    bits: every group's tiles are written and read back in the same order."""
    if name == "small":
        b = _small_batch(21, 1024, n_roots=4, len_hi=160, ms=16)
        Hq, Hkv = heads
    else:
        b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    out, info, ref = pack_both(b)
    R, T = info["n_rows"], b.row_len
    shape = (W.AttnShape(R, T, Hq, Hkv, 128, "bf16", 128 ** -0.5, 0.5) if name == "small"
             else W.attn_shape(name, R, T))
    q, k, v, do = W.attn_tensors(shape, 7)
    g = GpuRun(out["subtree_end"], shape.n_q_heads, shape.n_kv_heads, 128, stp.STP_BF16, shape.scale,
               q, k, v, do).run()
    base = [x.clone() for x in (g.dq, g.dk, g.dv)]
    full_ws = g.buf.bwd_ws.numel()
    for dg in ds_groups:
        g.desc = stp.Desc(R, T, shape.n_q_heads, shape.n_kv_heads, 128, stp.STP_BF16, shape.scale,
                          g.desc.max_tile_pairs, ds_groups=dg)
        ws = torch.empty(stp.stp_workspace_size(g.desc)[2], dtype=torch.uint8, device="cuda")
        assert ws.numel() < full_ws
        for x in (g.dq, g.dk, g.dv):
            x.fill_(float("nan"))
        stp.stp_attn_bwd(g.desc, g.q, g.k, g.v, g.o, g.lse, g.do, g.se, g.buf.tile_meta, g.dq, g.dk, g.dv, ws)
        torch.cuda.synchronize()
        assert stp.stp_device_status(ws) == stp.STP_OK
        for got, want in zip((g.dq, g.dk, g.dv), base):
            assert torch.equal(got, want), dg
