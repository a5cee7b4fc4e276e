"""stp_classify_noalloc: the classification entry point for callers that
cannot allocate device memory (graph capture, plug-in hosts that only pass
their input and output buffers).  It must give exactly what stp_classify
gives, also on back-to-back calls that reuse the library's fixed scratch.

Kept in its own file, collected last, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from gpu_helpers import pack_both
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(desc, se):
    """Tile classes and forward outputs from both entry points."""
    R, T = desc.n_rows, desc.row_len
    nt = T // 128
    out = {}
    q = torch.randn(R, T, desc.n_q_heads, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    k = torch.randn(R, T, desc.n_kv_heads, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    v = torch.randn(R, T, desc.n_kv_heads, 128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    for name, fn in (("alloc", stp.stp_classify), ("noalloc", stp.stp_classify_noalloc)):
        buf = stp.Buffers(desc)
        fn(desc, se, buf.tile_meta)
        cls = torch.empty(R, nt, nt, dtype=torch.int8, device="cuda")
        stp.stp_read_tile_classes(desc, buf.tile_meta, cls)
        o = torch.empty_like(q)
        lse = torch.empty(R, desc.n_q_heads, T, dtype=torch.float32, device="cuda")
        stp.stp_attn_fwd(desc, q, k, v, se, buf.tile_meta, o, lse, buf.fwd_ws)
        torch.cuda.synchronize()
        assert stp.stp_device_status(buf.tile_meta) == stp.STP_OK
        out[name] = (cls.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy())
    return out


def _desc_for(b):
    out, info, _ = pack_both(b)
    se = torch.from_numpy(out["subtree_end"]).cuda()
    return stp.Desc(info["n_rows"], b.row_len, 4, 2, 128, stp.STP_BF16), se


def test_noalloc_matches_classify_on_two_calls_in_a_row(stp_lib):
    # two different batches back to back: the second call reuses the scratch
    # the first one left behind
    for b in (W.curriculum(2), W.grpo(1)):
        desc, se = _desc_for(b)
        res = _run(desc, se)
        np.testing.assert_array_equal(res["noalloc"][0], res["alloc"][0])
        # the work lists drive the forward: identical lists, identical outputs
        np.testing.assert_array_equal(res["noalloc"][1], res["alloc"][1])
        np.testing.assert_array_equal(res["noalloc"][2], res["alloc"][2])


def test_noalloc_rejects_sizes_beyond_its_scratch(stp_lib):
    desc = stp.Desc(129, 131072, 1, 1, 128, stp.STP_BF16)   # 129 x 1024 tiles > 131072
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    meta = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(stp.StpError) as e:
        stp.stp_classify_noalloc(desc, x, meta)
    assert e.value.status == stp.STP_EINVAL
    assert "scratch" in str(e.value)
