"""Shared helpers of the GPU tests: run the product path through the C ABI
(C++ packer -> device classify -> fwd -> bwd) and the oracle on the same
seeded inputs."""
import numpy as np
import torch

from oracle import pack as OP
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W

BF16_TOL = {"o": 1e-2, "lse": 1e-3, "grad_rel": 2e-2}
FP32_TOL = 1e-5


def pack_both(b):
    """(C++ plan arrays + info, oracle plan) for a batch."""
    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len,
                        min_shared=b.min_shared)
    out = stp.stp_plan_write(plan)
    info = stp.stp_plan_info(plan)
    ref = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
    return out, info, ref


class GpuRun:
    """Device buffers and one classify + fwd (+ bwd) pass through the C ABI."""

    def __init__(self, subtree_end: np.ndarray, n_q_heads, n_kv_heads, head_dim, dtype, scale,
                 q, k, v, do=None):
        R, T = subtree_end.shape
        try:  # size the backward's dS workspace exactly when subtree_end is valid
            pairs = stp.stp_count_tile_pairs(subtree_end) if R > 0 else 0
        except stp.StpError:
            pairs = 0
        self.desc = stp.Desc(R, T, n_q_heads, n_kv_heads, head_dim, dtype, scale, pairs)
        self.buf = stp.Buffers(self.desc)
        dev = "cuda"
        self.se = torch.from_numpy(np.ascontiguousarray(subtree_end)).to(dev)
        self.q, self.k, self.v = (x.to(dev).contiguous() for x in (q, k, v))
        self.do = None if do is None else do.to(dev).contiguous()
        tdt = self.q.dtype
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(R, n_q_heads, T, dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        assert tdt == (torch.bfloat16 if dtype == stp.STP_BF16 else torch.float32)

    def classify(self):
        stp.stp_classify(self.desc, self.se, self.buf.tile_meta)

    def tile_classes(self):
        R, T = self.desc.n_rows, self.desc.row_len
        nt = T // 128
        cls = torch.empty(R, nt, nt, dtype=torch.int8, device="cuda")
        stp.stp_read_tile_classes(self.desc, self.buf.tile_meta, cls)
        torch.cuda.synchronize()
        return cls.cpu().numpy()

    def fwd(self):
        stp.stp_attn_fwd(self.desc, self.q, self.k, self.v, self.se, self.buf.tile_meta, self.o,
                         self.lse, self.buf.fwd_ws)

    def bwd(self):
        stp.stp_attn_bwd(self.desc, self.q, self.k, self.v, self.o, self.lse, self.do, self.se,
                         self.buf.tile_meta, self.dq, self.dk, self.dv, self.buf.bwd_ws)

    def run(self, backward=True):
        self.classify()
        self.fwd()
        if backward:
            self.bwd()
        torch.cuda.synchronize()
        assert stp.stp_device_status(self.buf.tile_meta) == stp.STP_OK
        assert stp.stp_device_status(self.buf.fwd_ws) == stp.STP_OK
        if backward:
            assert stp.stp_device_status(self.buf.bwd_ws) == stp.STP_OK
        return self


def tensors_for(shape: W.AttnShape, seed):
    return W.attn_tensors(shape, seed)


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))
