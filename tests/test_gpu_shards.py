"""Sharding by (row, kv head): launching each shard separately and putting
the pieces together gives the full launch's results.  Rows and kv-head
groups share nothing, so O, LSE, dK and dV are bit-identical; dQ is summed
with float reductions whose order varies from run to run, so it is compared
with the usual bf16 gradient tolerance.  On a one-GPU machine the shards of all
ranks run one after another."""
import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, GpuRun, pack_both, rel_err
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W
from sft_trie_build_gb300.shard import shard_units, unit_runs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
def test_shards_reassemble_full_launch(stp_lib, world):
    b = W.curriculum(2)
    out, info, _ = pack_both(b)
    se = out["subtree_end"]
    R, T = info["n_rows"], b.row_len
    shape = W.attn_shape("curriculum", R, T)
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    G = Hq // Hkv
    q, k, v, do = W.attn_tensors(shape, 5)
    full = GpuRun(se, Hq, Hkv, 128, stp.STP_BF16, shape.scale, q, k, v, do).run()
    fo, fl, fdq, fdk, fdv = (x.cpu() for x in (full.o, full.lse, full.dq, full.dk, full.dv))
    dq_parts, dq_full = [], []
    for rank in range(world):
        u0, u1 = shard_units(R, Hkv, world, rank)
        for r, g0, g1 in unit_runs(u0, u1, Hkv):
            hq = slice(g0 * G, g1 * G)
            part = GpuRun(se[r:r + 1], (g1 - g0) * G, g1 - g0, 128, stp.STP_BF16, shape.scale,
                          q[r:r + 1, :, hq], k[r:r + 1, :, g0:g1], v[r:r + 1, :, g0:g1],
                          do[r:r + 1, :, hq]).run()
            assert torch.equal(part.o.cpu(), fo[r:r + 1, :, hq])
            assert torch.equal(part.lse.cpu(), fl[r:r + 1, hq])
            assert torch.equal(part.dk.cpu(), fdk[r:r + 1, :, g0:g1])
            assert torch.equal(part.dv.cpu(), fdv[r:r + 1, :, g0:g1])
            dq_parts.append(part.dq.float().cpu().numpy())
            dq_full.append(fdq[r:r + 1, :, hq].float().numpy())
    assert rel_err(np.concatenate([x.ravel() for x in dq_parts]),
                   np.concatenate([x.ravel() for x in dq_full])) <= BF16_TOL["grad_rel"]
