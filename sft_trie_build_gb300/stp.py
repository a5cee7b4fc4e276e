"""Python binding of libstp.so (include/stp.h): the same entry points, with
argument marshalling only.  Every step of the path runs in the library: the
host packer in C++, classification and attention in CUDA kernels.  There is
no fallback: if the library is missing or a call fails, an exception says so.

Device tensors are torch CUDA tensors (PyTorch only provides device memory and
streams); host arrays are numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libstp.so")

STP_OK, STP_EINVAL, STP_ETOOLONG, STP_ENOMEM, STP_ECUDA, STP_EUNSUPPORTED, STP_EDEVICE = range(7)
STATUS_NAMES = {0: "STP_OK", 1: "STP_EINVAL", 2: "STP_ETOOLONG", 3: "STP_ENOMEM", 4: "STP_ECUDA",
                5: "STP_EUNSUPPORTED", 6: "STP_EDEVICE"}
STP_GLOBAL, STP_PER_FAMILY, STP_IN_ORDER = 0, 1, 2
STP_BF16, STP_FP32 = 0, 1

EXPORTED = ["stp_pack", "stp_plan_info", "stp_plan_write", "stp_plan_rows_of", "stp_plan_times", "stp_plan_free",
            "stp_plan_rows", "stp_plan_rows_many",
            "stp_count_tile_pairs", "stp_workspace_size", "stp_classify", "stp_classify_noalloc", "stp_read_tile_classes",
            "stp_attn_fwd", "stp_attn_bwd", "stp_step_scratch_size", "stp_attn_step_host",
            "stp_index_workspace_size", "stp_index_topk",
            "stp_logprob_workspace_size", "stp_logprob_gather",
            "stp_gdn_plan_bound", "stp_gdn_plan", "stp_gdn_workspace_size", "stp_gdn_fwd",
            "stp_gdn_train_workspace_size", "stp_gdn_fwd_train", "stp_gdn_bwd",
            "stp_device_status", "stp_last_error", "stp_version"]


class StpError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("row_len", ctypes.c_int32),
                ("input_tokens", ctypes.c_int64), ("packed_tokens", ctypes.c_int64),
                ("n_segments", ctypes.c_int64), ("n_leaves", ctypes.c_int64),
                ("useful_pairs", ctypes.c_int64), ("tree_token_ratio", ctypes.c_double)]


class IndexDesc(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("row_len", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("top_k", ctypes.c_int32), ("max_tile_pairs", ctypes.c_int32)]


class LogprobDesc(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("row_len", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("vocab", ctypes.c_int32)]


class GdnDesc(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("row_len", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("row_len", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("max_tile_pairs", ctypes.c_int32), ("ds_groups", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_U8P = ctypes.POINTER(ctypes.c_uint8)
_SZ = ctypes.POINTER(ctypes.c_size_t)


def lib():
    """Loads libstp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with sft_trie_build_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        st = ctypes.c_int32
        L.stp_pack.argtypes = [_I32P, _I64P, ctypes.c_int32, _U8P, _I32P, ctypes.c_int32,
                               ctypes.c_int32, ctypes.c_uint32, ctypes.POINTER(_P)]
        L.stp_pack.restype = st
        L.stp_plan_info.argtypes = [_P, ctypes.POINTER(PlanInfo)]
        L.stp_plan_info.restype = st
        L.stp_plan_write.argtypes = [_P, _I32P, _I32P, _I32P, _U8P, _I64P]
        L.stp_plan_write.restype = st
        L.stp_plan_rows_of.argtypes = [_P, _I32P]
        L.stp_plan_rows_of.restype = st
        L.stp_plan_times.argtypes = [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        L.stp_plan_times.restype = st
        L.stp_plan_free.argtypes = [_P]
        L.stp_plan_free.restype = None
        L.stp_plan_rows.argtypes = [_I32P, _I64P, ctypes.c_int32, _U8P, _I32P, _I32P, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, _I32P, _I64P]
        L.stp_plan_rows.restype = st
        L.stp_plan_rows_many.argtypes = [_I32P, _I64P, ctypes.c_int32, _U8P, _I32P, _I32P, _I64P,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32,
                                         ctypes.c_int32, _I32P, _I64P]
        L.stp_plan_rows_many.restype = st
        L.stp_count_tile_pairs.argtypes = [_I32P, ctypes.c_int32, ctypes.c_int32, _I64P]
        L.stp_count_tile_pairs.restype = st
        L.stp_workspace_size.argtypes = [ctypes.POINTER(AttnDesc), _SZ, _SZ, _SZ]
        L.stp_workspace_size.restype = st
        L.stp_classify.argtypes = [ctypes.POINTER(AttnDesc), _P, _P, _P]
        L.stp_classify.restype = st
        L.stp_classify_noalloc.argtypes = [ctypes.POINTER(AttnDesc), _P, _P, _P]
        L.stp_classify_noalloc.restype = st
        L.stp_read_tile_classes.argtypes = [ctypes.POINTER(AttnDesc), _P, _P, _P]
        L.stp_read_tile_classes.restype = st
        L.stp_attn_fwd.argtypes = [ctypes.POINTER(AttnDesc), _P, _P, _P, _P, _P, _P, _P, _P, _P]
        L.stp_attn_fwd.restype = st
        L.stp_attn_bwd.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 13
        L.stp_attn_bwd.restype = st
        L.stp_step_scratch_size.argtypes = [ctypes.POINTER(AttnDesc), ctypes.c_int32, _SZ]
        L.stp_step_scratch_size.restype = st
        L.stp_attn_step_host.argtypes = [ctypes.POINTER(AttnDesc), ctypes.c_int32] + [_P] * 12 + \
            [ctypes.c_size_t, _P]
        L.stp_attn_step_host.restype = st
        L.stp_index_workspace_size.argtypes = [ctypes.POINTER(IndexDesc), _SZ]
        L.stp_index_workspace_size.restype = st
        L.stp_index_topk.argtypes = [ctypes.POINTER(IndexDesc)] + [_P] * 9
        L.stp_index_topk.restype = st
        L.stp_logprob_workspace_size.argtypes = [ctypes.POINTER(LogprobDesc), _SZ]
        L.stp_logprob_workspace_size.restype = st
        L.stp_logprob_gather.argtypes = [ctypes.POINTER(LogprobDesc)] + [_P] * 7
        L.stp_logprob_gather.restype = st
        L.stp_gdn_plan_bound.argtypes = [ctypes.POINTER(GdnDesc), _SZ]
        L.stp_gdn_plan_bound.restype = st
        L.stp_gdn_plan.argtypes = [ctypes.POINTER(GdnDesc), _I32P, _I32P, _P, ctypes.c_size_t]
        L.stp_gdn_plan.restype = st
        L.stp_gdn_workspace_size.argtypes = [ctypes.POINTER(GdnDesc), _P, _SZ]
        L.stp_gdn_workspace_size.restype = st
        L.stp_gdn_fwd.argtypes = [ctypes.POINTER(GdnDesc)] + [_P] * 9
        L.stp_gdn_fwd.restype = st
        L.stp_gdn_train_workspace_size.argtypes = [ctypes.POINTER(GdnDesc), _P, _SZ]
        L.stp_gdn_train_workspace_size.restype = st
        L.stp_gdn_fwd_train.argtypes = [ctypes.POINTER(GdnDesc)] + [_P] * 9
        L.stp_gdn_fwd_train.restype = st
        L.stp_gdn_bwd.argtypes = [ctypes.POINTER(GdnDesc)] + [_P] * 13
        L.stp_gdn_bwd.restype = st
        L.stp_device_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int32)]
        L.stp_device_status.restype = st
        L.stp_last_error.argtypes = []
        L.stp_last_error.restype = ctypes.c_char_p
        L.stp_version.argtypes = []
        L.stp_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status, where):
    if status != STP_OK:
        raise StpError(status, where, lib().stp_last_error().decode())


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def _dptr(t):
    """Device pointer of a torch tensor (or an int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------------------
# Host packer
# ---------------------------------------------------------------------------

class Plan:
    """Owns an stp_plan handle (freed with stp_plan_free)."""

    def __init__(self, handle, n_seqs, n_tokens):
        self.handle = handle
        self.n_seqs = n_seqs
        self.n_tokens = n_tokens

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.stp_plan_free(h)
            self.handle = None


def stp_pack(tokens: np.ndarray, offsets: np.ndarray, trainable=None, family=None, *,
             row_len: int, min_shared: int = 64, flags: int = STP_GLOBAL) -> Plan:
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    n = len(offsets) - 1
    tr = None if trainable is None else np.ascontiguousarray(trainable, dtype=np.uint8)
    fam = None if family is None else np.ascontiguousarray(family, dtype=np.int32)
    h = _P()
    _check(lib().stp_pack(_ptr(tokens, ctypes.c_int32), _ptr(offsets, ctypes.c_int64), n,
                          _ptr(tr, ctypes.c_uint8), _ptr(fam, ctypes.c_int32), int(row_len),
                          int(min_shared), int(flags), ctypes.byref(h)), "stp_pack")
    return Plan(h, n, int(offsets[-1]) if n > 0 else 0)


def stp_plan_info(plan: Plan) -> dict:
    info = PlanInfo()
    _check(lib().stp_plan_info(plan.handle, ctypes.byref(info)), "stp_plan_info")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


def stp_plan_write(plan: Plan, out=None) -> dict:
    """Materializes the plan into host arrays (allocated here when ``out`` is
    None; pass a dict of preallocated, e.g. pinned, arrays to reuse them)."""
    info = stp_plan_info(plan)
    R, T = info["n_rows"], info["row_len"]
    if out is None:
        out = {"token_ids": np.empty((R, T), np.int32), "position_ids": np.empty((R, T), np.int32),
               "subtree_end": np.empty((R, T), np.int32), "loss_mask": np.empty((R, T), np.uint8),
               "gather_index": np.empty(plan.n_tokens, np.int64)}
    _check(lib().stp_plan_write(plan.handle, _ptr(out.get("token_ids"), ctypes.c_int32),
                                _ptr(out.get("position_ids"), ctypes.c_int32),
                                _ptr(out.get("subtree_end"), ctypes.c_int32),
                                _ptr(out.get("loss_mask"), ctypes.c_uint8),
                                _ptr(out.get("gather_index"), ctypes.c_int64)), "stp_plan_write")
    return out


def stp_plan_times(plan: Plan) -> dict:
    """Host milliseconds stp_pack spent on the trie walk and on the placement."""
    w, p = ctypes.c_double(), ctypes.c_double()
    _check(lib().stp_plan_times(plan.handle, ctypes.byref(w), ctypes.byref(p)), "stp_plan_times")
    return {"walk_ms": w.value, "place_ms": p.value}


def stp_plan_rows_of(plan: Plan) -> np.ndarray:
    out = np.empty(plan.n_seqs, np.int32)
    _check(lib().stp_plan_rows_of(plan.handle, _ptr(out, ctypes.c_int32)), "stp_plan_rows_of")
    return out


# ---------------------------------------------------------------------------
# Device calls
# ---------------------------------------------------------------------------

@dataclass
class Desc:
    n_rows: int
    row_len: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: int = STP_BF16
    scale: float = 0.0
    max_tile_pairs: int = 0   # 0 = every lower-triangular tile pair
    ds_groups: int = 0        # kv-head groups whose dS tiles the backward holds at once (0 = all)

    def c(self) -> AttnDesc:
        sc = self.scale if self.scale > 0 else self.head_dim ** -0.5
        return AttnDesc(self.n_rows, self.row_len, self.n_q_heads, self.n_kv_heads, self.head_dim,
                        self.dtype, sc, 128, 128, self.max_tile_pairs, self.ds_groups)


def _pool(tokens, offsets, trainable, family):
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    tr = None if trainable is None else np.ascontiguousarray(trainable, dtype=np.uint8)
    fam = None if family is None else np.ascontiguousarray(family, dtype=np.int32)
    return tokens, offsets, tr, fam


def stp_plan_rows(tokens, offsets, trainable=None, family=None, subset=None, *, row_len: int,
                  min_shared: int = 64, flags: int = STP_GLOBAL):
    """(rows, packed tokens) that packing pool[subset] would give, without a plan."""
    tokens, offsets, tr, fam = _pool(tokens, offsets, trainable, family)
    sub = None if subset is None else np.ascontiguousarray(subset, dtype=np.int32)
    r, pk = ctypes.c_int32(), ctypes.c_int64()
    _check(lib().stp_plan_rows(_ptr(tokens, ctypes.c_int32), _ptr(offsets, ctypes.c_int64), len(offsets) - 1,
                               _ptr(tr, ctypes.c_uint8), _ptr(fam, ctypes.c_int32), _ptr(sub, ctypes.c_int32),
                               0 if sub is None else len(sub), int(row_len), int(min_shared), int(flags),
                               ctypes.byref(r), ctypes.byref(pk)), "stp_plan_rows")
    return r.value, pk.value


def stp_plan_rows_many(tokens, offsets, trainable=None, family=None, subsets=(), *, row_len: int,
                       min_shared: int = 64, flags: int = STP_GLOBAL, n_threads: int = 0):
    """stp_plan_rows over a list of index arrays, planned in parallel on host threads."""
    tokens, offsets, tr, fam = _pool(tokens, offsets, trainable, family)
    subs = [np.ascontiguousarray(s, dtype=np.int32) for s in subsets]
    so = np.zeros(len(subs) + 1, np.int64)
    so[1:] = np.cumsum([len(s) for s in subs])
    flat = np.concatenate(subs) if subs else np.zeros(0, np.int32)
    rows = np.zeros(len(subs), np.int32)
    packed = np.zeros(len(subs), np.int64)
    if subs:
        _check(lib().stp_plan_rows_many(_ptr(tokens, ctypes.c_int32), _ptr(offsets, ctypes.c_int64),
                                        len(offsets) - 1, _ptr(tr, ctypes.c_uint8), _ptr(fam, ctypes.c_int32),
                                        _ptr(flat, ctypes.c_int32), _ptr(so, ctypes.c_int64), len(subs),
                                        int(row_len), int(min_shared), int(flags), int(n_threads),
                                        _ptr(rows, ctypes.c_int32), _ptr(packed, ctypes.c_int64)),
               "stp_plan_rows_many")
    return rows, packed


def stp_count_tile_pairs(subtree_end: np.ndarray) -> int:
    """Exact non-empty (query tile, key tile) pairs of a host int32 [R, T] subtree_end."""
    se = np.ascontiguousarray(subtree_end, dtype=np.int32)
    if se.ndim != 2:
        raise ValueError("subtree_end must be [n_rows, row_len]")
    out = ctypes.c_int64()
    _check(lib().stp_count_tile_pairs(_ptr(se, ctypes.c_int32), se.shape[0], se.shape[1], ctypes.byref(out)),
           "stp_count_tile_pairs")
    return out.value


def stp_workspace_size(desc: Desc):
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    d = desc.c()
    _check(lib().stp_workspace_size(ctypes.byref(d), ctypes.byref(a), ctypes.byref(b),
                                    ctypes.byref(c)), "stp_workspace_size")
    return a.value, b.value, c.value


def stp_classify(desc: Desc, subtree_end, tile_meta, stream=None):
    d = desc.c()
    _check(lib().stp_classify(ctypes.byref(d), _dptr(subtree_end), _dptr(tile_meta), _stream(stream)),
           "stp_classify")


def stp_classify_noalloc(desc: Desc, subtree_end, tile_meta, stream=None):
    """stp_classify without device allocation: scratch lives in the library's
    fixed 1 MiB device array (at most 131072 tiles; calls overlapping on the
    GPU race).  Make the first call on a device before any stream capture."""
    d = desc.c()
    _check(lib().stp_classify_noalloc(ctypes.byref(d), _dptr(subtree_end), _dptr(tile_meta),
                                      _stream(stream)), "stp_classify_noalloc")


def stp_read_tile_classes(desc: Desc, tile_meta, cls_out, stream=None):
    d = desc.c()
    _check(lib().stp_read_tile_classes(ctypes.byref(d), _dptr(tile_meta), _dptr(cls_out),
                                       _stream(stream)), "stp_read_tile_classes")


def stp_attn_fwd(desc: Desc, q, k, v, subtree_end, tile_meta, o, lse, ws, stream=None):
    d = desc.c()
    _check(lib().stp_attn_fwd(ctypes.byref(d), _dptr(q), _dptr(k), _dptr(v), _dptr(subtree_end),
                              _dptr(tile_meta), _dptr(o), _dptr(lse), _dptr(ws), _stream(stream)),
           "stp_attn_fwd")


def stp_attn_bwd(desc: Desc, q, k, v, o, lse, d_o, subtree_end, tile_meta, dq, dk, dv, ws,
                 stream=None):
    d = desc.c()
    _check(lib().stp_attn_bwd(ctypes.byref(d), _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse),
                              _dptr(d_o), _dptr(subtree_end), _dptr(tile_meta), _dptr(dq),
                              _dptr(dk), _dptr(dv), _dptr(ws), _stream(stream)), "stp_attn_bwd")


def stp_step_scratch_size(desc: Desc, n_chunks: int) -> int:
    out = ctypes.c_size_t()
    d = desc.c()
    _check(lib().stp_step_scratch_size(ctypes.byref(d), n_chunks, ctypes.byref(out)),
           "stp_step_scratch_size")
    return out.value


def stp_attn_step_host(desc: Desc, n_chunks: int, q, k, v, d_o, subtree_end, tile_meta,
                       o, lse, dq, dk, dv, scratch, stream=None):
    """Forward + backward on host tensors (torch CPU tensors, ideally pinned):
    q, k, v, d_o in; o, lse, dq, dk, dv out.  subtree_end, tile_meta and
    scratch are device tensors.  Outputs are valid once `stream` is synced."""
    for t in (q, k, v, d_o, o, lse, dq, dk, dv):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("stp_attn_step_host takes contiguous host tensors")
    d = desc.c()
    _check(lib().stp_attn_step_host(ctypes.byref(d), n_chunks, _dptr(q), _dptr(k), _dptr(v), _dptr(d_o),
                                    _dptr(subtree_end), _dptr(tile_meta), _dptr(o), _dptr(lse),
                                    _dptr(dq), _dptr(dk), _dptr(dv), _dptr(scratch),
                                    scratch.numel() * scratch.element_size(), _stream(stream)),
           "stp_attn_step_host")


def index_desc(n_rows, row_len, n_heads, head_dim, top_k, max_tile_pairs=0) -> IndexDesc:
    return IndexDesc(n_rows, row_len, n_heads, head_dim, top_k, max_tile_pairs)


def stp_index_workspace_size(desc: IndexDesc) -> int:
    out = ctypes.c_size_t()
    _check(lib().stp_index_workspace_size(ctypes.byref(desc), ctypes.byref(out)), "stp_index_workspace_size")
    return out.value


def stp_index_topk(desc: IndexDesc, q, k, w, subtree_end, tile_meta, topk_idx, topk_score, ws, stream=None):
    _check(lib().stp_index_topk(ctypes.byref(desc), _dptr(q), _dptr(k), _dptr(w), _dptr(subtree_end),
                                _dptr(tile_meta), _dptr(topk_idx), _dptr(topk_score), _dptr(ws), _stream(stream)),
           "stp_index_topk")


def logprob_desc(n_rows, row_len, hidden, vocab) -> LogprobDesc:
    return LogprobDesc(n_rows, row_len, hidden, vocab)


def stp_logprob_workspace_size(desc: LogprobDesc) -> int:
    out = ctypes.c_size_t()
    _check(lib().stp_logprob_workspace_size(ctypes.byref(desc), ctypes.byref(out)), "stp_logprob_workspace_size")
    return out.value


def stp_logprob_gather(desc: LogprobDesc, hidden, w_vocab, token_ids, loss_mask, logprob, ws, stream=None):
    _check(lib().stp_logprob_gather(ctypes.byref(desc), _dptr(hidden), _dptr(w_vocab), _dptr(token_ids),
                                    _dptr(loss_mask), _dptr(logprob), _dptr(ws), _stream(stream)),
           "stp_logprob_gather")


# plan header fields (int32 words), as the library writes them
GP_MAGIC, GP_N, GP_NSEG, GP_NCHUNK, GP_NDEPTH, GP_WORDS, GP_PREV, GP_SEG_START, GP_SEG_LEN, GP_SEG_PARENT, \
    GP_SEG_CHUNK0, GP_DEPTH_OFF, GP_CHUNK_START, GP_CHUNK_LEN, GP_MAX_DEPTH_SEGS, GP_PREV2, GP_PREV3, \
    GP_CHILD_OFF, GP_CHILD, GP_SUCC_OFF, GP_SUCC = range(21)


def gdn_desc(n_rows, row_len, n_heads, head_dim=128, scale=None) -> GdnDesc:
    return GdnDesc(n_rows, row_len, n_heads, head_dim, head_dim ** -0.5 if scale is None else scale)


def stp_gdn_plan_bound(desc: GdnDesc) -> int:
    out = ctypes.c_size_t()
    _check(lib().stp_gdn_plan_bound(ctypes.byref(desc), ctypes.byref(out)), "stp_gdn_plan_bound")
    return out.value


def stp_gdn_plan(desc: GdnDesc, subtree_end: np.ndarray, row_used=None) -> np.ndarray:
    """Host plan (int32 words, trimmed to the words used) of the tree-aware GDN."""
    se = np.ascontiguousarray(subtree_end, dtype=np.int32)
    used = None if row_used is None else np.ascontiguousarray(row_used, dtype=np.int32)
    nbytes = stp_gdn_plan_bound(desc)
    buf = np.zeros(nbytes // 4, np.int32)
    _check(lib().stp_gdn_plan(ctypes.byref(desc), _ptr(se, ctypes.c_int32), _ptr(used, ctypes.c_int32),
                              buf.ctypes.data_as(_P), nbytes), "stp_gdn_plan")
    return buf[: buf[GP_WORDS]].copy()


def gdn_plan_arrays(plan: np.ndarray) -> dict:
    """Named views of a host plan's arrays."""
    w = plan
    n, ns, nc, nd = w[GP_N], w[GP_NSEG], w[GP_NCHUNK], w[GP_NDEPTH]
    at = lambda f, k: w[w[f]: w[f] + k]  # noqa: E731
    return {"prev": at(GP_PREV, n), "prev2": at(GP_PREV2, n), "prev3": at(GP_PREV3, n), "seg_start": at(GP_SEG_START, ns), "seg_len": at(GP_SEG_LEN, ns),
            "seg_parent": at(GP_SEG_PARENT, ns), "seg_chunk0": at(GP_SEG_CHUNK0, ns),
            "depth_off": at(GP_DEPTH_OFF, nd + 1), "chunk_start": at(GP_CHUNK_START, nc),
            "chunk_len": at(GP_CHUNK_LEN, nc), "child_off": at(GP_CHILD_OFF, ns + 1),
            "child": at(GP_CHILD, w[w[GP_CHILD_OFF] + ns] if ns > 0 else 0),
            "succ_off": at(GP_SUCC_OFF, n + 1), "succ": at(GP_SUCC, w[w[GP_SUCC_OFF] + n] if n > 0 else 0)}


def stp_gdn_workspace_size(desc: GdnDesc, plan: np.ndarray) -> int:
    out = ctypes.c_size_t()
    _check(lib().stp_gdn_workspace_size(ctypes.byref(desc), plan.ctypes.data_as(_P), ctypes.byref(out)),
           "stp_gdn_workspace_size")
    return out.value


def stp_gdn_fwd(desc: GdnDesc, plan: np.ndarray, d_plan, x, conv_w, g, beta, o, ws, stream=None):
    _check(lib().stp_gdn_fwd(ctypes.byref(desc), plan.ctypes.data_as(_P), _dptr(d_plan), _dptr(x),
                             _dptr(conv_w), _dptr(g), _dptr(beta), _dptr(o), _dptr(ws), _stream(stream)),
           "stp_gdn_fwd")


def stp_gdn_train_workspace_size(desc: GdnDesc, plan: np.ndarray) -> int:
    out = ctypes.c_size_t()
    _check(lib().stp_gdn_train_workspace_size(ctypes.byref(desc), plan.ctypes.data_as(_P), ctypes.byref(out)),
           "stp_gdn_train_workspace_size")
    return out.value


def stp_gdn_fwd_train(desc: GdnDesc, plan: np.ndarray, d_plan, x, conv_w, g, beta, o, ws, stream=None):
    _check(lib().stp_gdn_fwd_train(ctypes.byref(desc), plan.ctypes.data_as(_P), _dptr(d_plan), _dptr(x),
                                   _dptr(conv_w), _dptr(g), _dptr(beta), _dptr(o), _dptr(ws), _stream(stream)),
           "stp_gdn_fwd_train")


def stp_gdn_bwd(desc: GdnDesc, plan: np.ndarray, d_plan, x, conv_w, g, beta, d_o, dx, dconv_w, dg, dbeta, ws,
                stream=None):
    _check(lib().stp_gdn_bwd(ctypes.byref(desc), plan.ctypes.data_as(_P), _dptr(d_plan), _dptr(x), _dptr(conv_w),
                             _dptr(g), _dptr(beta), _dptr(d_o), _dptr(dx), _dptr(dconv_w), _dptr(dg), _dptr(dbeta),
                             _dptr(ws), _stream(stream)), "stp_gdn_bwd")


def stp_device_status(ws, stream=None) -> int:
    out = ctypes.c_int32()
    _check(lib().stp_device_status(_dptr(ws), _stream(stream), ctypes.byref(out)),
           "stp_device_status")
    return out.value


def stp_version() -> str:
    return lib().stp_version().decode()


# ---------------------------------------------------------------------------
# Convenience: buffers for one descriptor
# ---------------------------------------------------------------------------

class Buffers:
    """Caller-owned device buffers (torch) for one attention descriptor."""

    def __init__(self, desc: Desc, device="cuda"):
        import torch
        meta, fwd, bwd = stp_workspace_size(desc)
        self.tile_meta = torch.empty(max(meta, 256), dtype=torch.uint8, device=device)
        self.fwd_ws = torch.empty(max(fwd, 256), dtype=torch.uint8, device=device)
        self.bwd_ws = torch.empty(max(bwd, 256), dtype=torch.uint8, device=device)
