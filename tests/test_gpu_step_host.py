"""The host-buffer step (stp_attn_step_host): upload, forward, backward and
download pipelined over groups of kv heads.  Groups share nothing, so O, LSE,
dK and dV equal the device calls on the whole problem bit for bit; dQ is
summed with float reductions whose order varies, so it gets the bf16 gradient
tolerance (float32: its own small bound).  The error paths are checked too."""
import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, GpuRun, pack_both, rel_err
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _step(g: GpuRun, n_chunks, pin=True):
    d = g.desc
    host = lambda t: (t.cpu().contiguous().pin_memory() if pin else t.cpu().contiguous())  # noqa: E731
    q, k, v, do = (host(x) for x in (g.q, g.k, g.v, g.do))
    o, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty(d.n_rows, d.n_q_heads, d.row_len, dtype=torch.float32)
    if pin:
        o, dq, dk, dv, lse = (x.pin_memory() for x in (o, dq, dk, dv, lse))
    scratch = torch.empty(stp.stp_step_scratch_size(d, n_chunks), dtype=torch.uint8, device="cuda")
    stp.stp_classify(d, g.se, g.buf.tile_meta)
    stp.stp_attn_step_host(d, n_chunks, q, k, v, do, g.se, g.buf.tile_meta, o, lse, dq, dk, dv, scratch)
    assert stp.stp_device_status(scratch) == stp.STP_OK
    return o, lse, dq, dk, dv


def _reference(name, seed):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    out, info, _ = pack_both(b)
    shape = W.attn_shape(name, info["n_rows"], b.row_len)
    q, k, v, do = W.attn_tensors(shape, seed)
    return GpuRun(out["subtree_end"], shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                  stp.STP_BF16, shape.scale, q, k, v, do).run()


@pytest.mark.parametrize("n_chunks", [1, 2, 4, 8])
def test_step_host_matches_device_calls(stp_lib, n_chunks):
    g = _reference("curriculum", 7)
    o, lse, dq, dk, dv = _step(g, n_chunks)
    assert torch.equal(o, g.o.cpu())
    assert torch.equal(lse, g.lse.cpu())
    assert torch.equal(dk, g.dk.cpu())
    assert torch.equal(dv, g.dv.cpu())
    assert rel_err(dq.float().numpy(), g.dq.float().cpu().numpy()) <= BF16_TOL["grad_rel"]


def test_step_host_grpo_row_and_repeat(stp_lib):
    """One 16384-token row; two steps in a row reuse the library's streams."""
    g = _reference("grpo", 3)
    for _ in range(2):
        o, lse, dq, dk, dv = _step(g, 4)
        assert torch.equal(o, g.o.cpu()) and torch.equal(lse, g.lse.cpu())
        assert torch.equal(dk, g.dk.cpu()) and torch.equal(dv, g.dv.cpu())
        assert rel_err(dq.float().numpy(), g.dq.float().cpu().numpy()) <= BF16_TOL["grad_rel"]


def test_step_host_fp32_pageable(stp_lib):
    """float32 path, ordinary (pageable) host memory."""
    b = W.random_forest(4, n_roots=3, max_depth=3, max_children=3, len_lo=8, len_hi=120,
                        row_len=512, min_shared=16, vocab=W.VOCAB)
    out, info, _ = pack_both(b)
    shape = W.AttnShape(info["n_rows"], 512, 4, 2, 64, "fp32", 0.125, 1.0)
    q, k, v, do = W.attn_tensors(shape, 2)
    g = GpuRun(out["subtree_end"], 4, 2, 64, stp.STP_FP32, 0.125, q, k, v, do).run()
    o, lse, dq, dk, dv = _step(g, 2, pin=False)
    assert torch.equal(o, g.o.cpu()) and torch.equal(lse, g.lse.cpu())
    assert torch.equal(dk, g.dk.cpu()) and torch.equal(dv, g.dv.cpu())
    assert np.abs(dq.numpy() - g.dq.cpu().numpy()).max() <= 1e-5


def test_step_host_errors(stp_lib):
    d = stp.Desc(1, 256, 4, 2, 128, stp.STP_BF16)
    with pytest.raises(stp.StpError) as e:
        stp.stp_step_scratch_size(d, 3)
    assert e.value.status == stp.STP_EINVAL
    need = stp.stp_step_scratch_size(d, 2)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, 4, 128, dtype=torch.bfloat16)
    kx = torch.zeros(256, 2, 128, dtype=torch.bfloat16)
    lse = torch.zeros(1, 4, 256)
    se = torch.arange(256, dtype=torch.int32, device="cuda")
    buf = stp.Buffers(d)
    stp.stp_classify(d, se, buf.tile_meta)
    with pytest.raises(stp.StpError) as e:
        stp.stp_attn_step_host(d, 2, x, kx, kx, x, se, buf.tile_meta, x, lse, x, kx, kx, small)
    assert e.value.status == stp.STP_EINVAL
    with pytest.raises(ValueError):
        stp.stp_attn_step_host(d, 2, x.cuda(), kx, kx, x, se, buf.tile_meta, x, lse, x, kx, kx, small)
