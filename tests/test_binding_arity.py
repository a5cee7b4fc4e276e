"""Every binding of a call that takes a descriptor reaches the library with
the right number of arguments: given a descriptor the library rejects, the
call raises StpError (the library's own check), never a TypeError from
argument marshalling.  No GPU is touched (stream 0, no device pointers)."""
import numpy as np
import pytest

from sft_trie_build_gb300 import stp


def test_attention_calls():
    bad = stp.Desc(1, 100, 1, 1, 64, stp.STP_BF16, 0.1)   # row_len not a multiple of 128
    with pytest.raises(stp.StpError):
        stp.stp_workspace_size(bad)
    with pytest.raises(stp.StpError):
        stp.stp_classify(bad, None, None, stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_classify_noalloc(bad, None, None, stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_attn_fwd(bad, None, None, None, None, None, None, None, None, stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_attn_bwd(bad, *([None] * 12), stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_step_scratch_size(bad, 8)
    with pytest.raises(stp.StpError):
        stp.stp_read_tile_classes(bad, None, None, stream=0)


def test_index_calls():
    bad = stp.index_desc(1, 100, 1, 64, 8)
    with pytest.raises(stp.StpError):
        stp.stp_index_workspace_size(bad)
    with pytest.raises(stp.StpError):
        stp.stp_index_topk(bad, None, None, None, None, None, None, None, None, stream=0)


def test_logprob_calls():
    bad = stp.logprob_desc(1, 100, 64, 10)
    with pytest.raises(stp.StpError):
        stp.stp_logprob_workspace_size(bad)
    with pytest.raises(stp.StpError):
        stp.stp_logprob_gather(bad, None, None, None, None, None, None, stream=0)


def test_gdn_calls():
    desc = stp.gdn_desc(1, 8, 1)
    plan = stp.stp_gdn_plan(desc, np.arange(8, dtype=np.int32)[None])
    bad = stp.gdn_desc(1, 8, 1, head_dim=64)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_workspace_size(bad, plan)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_fwd(bad, plan, None, None, None, None, None, None, None, stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_train_workspace_size(bad, plan)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_fwd_train(bad, plan, None, None, None, None, None, None, None, stream=0)
    with pytest.raises(stp.StpError):
        stp.stp_gdn_bwd(bad, plan, *([None] * 11), stream=0)
    with pytest.raises(stp.StpError):   # a plan that is not one
        stp.stp_gdn_workspace_size(desc, np.zeros_like(plan))
