"""GPU path vs the oracle on every element, at the workloads' full sizes.

One classify + forward + backward launch over the whole packed batch (all
rows, all heads, the launch configuration the benchmark times), then the
float64 oracle, run one kv-head group at a time (its query heads with their
kv head: groups never mix, so this is the oracle of the whole problem split
by group), compared element by element:

* O <= 1e-2 and LSE <= 1e-3 max abs;
* dQ, dK, dV: max |diff| / max |oracle| <= 2e-2, per kv-head group (each
  group's part of the tensor against its own largest magnitude);

on the same bf16-rounded inputs upcast to float64.  Every kv-head group of
the GRPO row (its 5000-token prefix keys have the longest accumulations),
of the many-tiny-branches row (mostly partial tiles) and of the
global-tree batch (all its rows in one launch) is checked; the deep 32K row
checks its first kv-head group (the oracle needs about a minute per group
there).  Observed errors are printed.
"""
import numpy as np
import pytest

from gpu_helpers import BF16_TOL, GpuRun, pack_both
from oracle import attn as OA
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(stp_lib):
    return stp_lib


def _max_rel(got, want):
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))


@pytest.mark.parametrize("name,groups", [("grpo", None), ("bushy", None), ("curriculum", None),
                                         ("deep", (0,))])
def test_bf16_workload_every_element(name, groups):
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    out, info, ref = pack_both(b)
    R, T = info["n_rows"], b.row_len
    shape = W.attn_shape(name, R, T)
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    G = Hq // Hkv
    q, k, v, do = W.attn_tensors(shape, 0)
    g = GpuRun(out["subtree_end"], Hq, Hkv, shape.head_dim, stp.STP_BF16, shape.scale, q, k, v, do).run()
    o_g = g.o.float().cpu().numpy()
    lse_g = g.lse.cpu().numpy()
    dq_g = g.dq.float().cpu().numpy()
    dk_g = g.dk.float().cpu().numpy()
    dv_g = g.dv.float().cpu().numpy()
    del g
    errs = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for gg in (groups if groups is not None else range(Hkv)):
        hs = slice(gg * G, (gg + 1) * G)
        kv = slice(gg, gg + 1)
        dq, dk, dv, o, lse = OA.attn_bwd(ref, q[:, :, hs], k[:, :, kv], v[:, :, kv], do[:, :, hs], shape.scale)
        errs["o"] = max(errs["o"], float(np.abs(o_g[:, :, hs] - o).max()))
        errs["lse"] = max(errs["lse"], float(np.abs(lse_g[:, hs] - lse).max()))
        errs["dq"] = max(errs["dq"], _max_rel(dq_g[:, :, hs], dq))
        errs["dk"] = max(errs["dk"], _max_rel(dk_g[:, :, kv], dk))
        errs["dv"] = max(errs["dv"], _max_rel(dv_g[:, :, kv], dv))
    print(f"\n{name}: rows {R} x {T}, heads {Hq}/{Hkv}, groups checked "
          f"{'all' if groups is None else list(groups)}: {errs}")
    assert errs["o"] <= BF16_TOL["o"], errs
    assert errs["lse"] <= BF16_TOL["lse"], errs
    for n in ("dq", "dk", "dv"):
        assert errs[n] <= BF16_TOL["grad_rel"], (n, errs)
