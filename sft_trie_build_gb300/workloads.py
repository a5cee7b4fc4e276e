"""Seeded synthetic workloads for prefix-tree packing and tree attention.

This module only draws random numbers: token sequences, their trainable
masks, family ids, and the attention tensors Q, K, V and dO.  It holds none
of the packing, masking or attention arithmetic, so that the CPU oracle and
the CUDA path can both be fed from it without sharing any of the method.

Shapes follow the workloads the prefix-tree-packing pages describe:

* ``tiny``      -- 64-token shared prefix + 4 branches U[24,40], one 256 row.
* ``grpo``      -- 5000-token system prefix + 16 rollouts U[100,1000], one
                   16384 row (the CoreWeave "ART-Optimized Megatron" page,
                   "How close are we with the ideal theoretical gain?").
* ``curriculum``-- 350-token system prompt -> 3 task families x 300 ->
                   16 groups per family x U[100,400] prompt -> 8 completions
                   U[50,300], 4096-token rows (the prefix-tree-packing page,
                   "one tree per RL group" comparison).
* ``deep``      -- 8192 -> 4 x 2048 -> 4 x U[256,1024] -> 2 x U[64,512],
                   one 32768 row.
* ``bushy``     -- 1024-token prefix + 512 branches U[8,32] + independent
                   U[64,512] sequences until the row is full, one 16384 row.
* ``rollout32`` -- 32 rollouts in four groups of eight: a 4096-token root, a
                   12000-token group prefix and completions of 2000 / 2000 /
                   12000 / 7000 tokens (the prefix-tree-packing page, the
                   32-rollout table).

Every non-leaf level is non-trainable and every leaf level is trainable
(sharing stops at trainable tokens, so deeper trees need non-trainable
interior levels).  Siblings get distinct first tokens so that the drawn tree
is the tree the sequences form.  Integer lengths are inclusive uniform draws.

Fit rule for single-row workloads: a draw is accepted when the sum of the
drawn node lengths plus one token per leaf is at most the row length; else
the next seed is drawn.  This is a bound on the drawn design only (one extra
token per leaf covers any context token a branch may repeat), not a packing
computation.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

VOCAB = 32000


@dataclass
class SeqBatch:
    """A batch of tokenized sequences ready for packing."""

    seqs: List[np.ndarray]            # int32 token ids, one array per sequence
    trainable: List[np.ndarray]       # uint8, same lengths as seqs
    family: Optional[np.ndarray]      # int32 [n_seqs] or None
    row_len: int
    min_shared: int = 64
    seed: int = 0                     # the accepted seed
    info: dict = field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return len(self.seqs)

    def flat(self):
        """Concatenated (tokens int32, offsets int64, trainable uint8)."""
        lens = np.array([len(s) for s in self.seqs], dtype=np.int64)
        offsets = np.zeros(len(self.seqs) + 1, dtype=np.int64)
        np.cumsum(lens, out=offsets[1:])
        if self.seqs:
            tokens = np.concatenate(self.seqs).astype(np.int32)
            train = np.concatenate(self.trainable).astype(np.uint8)
        else:
            tokens = np.zeros(0, np.int32)
            train = np.zeros(0, np.uint8)
        return tokens, offsets, train


class _Node:
    __slots__ = ("length", "trainable", "children", "family", "tokens")

    def __init__(self, length, trainable, family=None):
        self.length = int(length)
        self.trainable = bool(trainable)
        self.children: List["_Node"] = []
        self.family = family
        self.tokens = None


def _fill_tokens(rng, node: _Node, sibling_firsts: set):
    toks = rng.integers(0, VOCAB, size=node.length, dtype=np.int64)
    if node.length > 0:
        while int(toks[0]) in sibling_firsts:
            toks[0] = rng.integers(0, VOCAB)
        sibling_firsts.add(int(toks[0]))
    node.tokens = toks.astype(np.int32)
    firsts: set = set()
    for c in node.children:
        _fill_tokens(rng, c, firsts)


def _paths(node: _Node, prefix_tok, prefix_tr, fam, out):
    tok = prefix_tok + [node.tokens]
    tr = prefix_tr + [np.full(node.length, 1 if node.trainable else 0, np.uint8)]
    f = node.family if node.family is not None else fam
    if not node.children:
        out.append((np.concatenate(tok), np.concatenate(tr), f))
        return
    for c in node.children:
        _paths(c, tok, tr, f, out)


def _design_size(node: _Node) -> int:
    return node.length + sum(_design_size(c) for c in node.children)


def _leaves(node: _Node) -> int:
    return 1 if not node.children else sum(_leaves(c) for c in node.children)


def _batch_from_roots(rng, roots, row_len, min_shared, seed, info):
    firsts: set = set()
    for r in roots:
        _fill_tokens(rng, r, firsts)
    out = []
    for r in roots:
        _paths(r, [], [], None, out)
    seqs = [o[0] for o in out]
    tr = [o[1] for o in out]
    fams = [o[2] for o in out]
    family = None if any(f is None for f in fams) else np.array(fams, np.int32)
    return SeqBatch(seqs, tr, family, row_len, min_shared, seed, info)


def _uniform(rng, lo, hi):
    return int(rng.integers(lo, hi + 1))


def tiny(seed: int = 0) -> SeqBatch:
    """64-token non-trainable prefix + 4 trainable branches U[24,40]; row 256."""
    rng = np.random.default_rng(seed)
    root = _Node(64, False, family=0)
    root.children = [_Node(_uniform(rng, 24, 40), True) for _ in range(4)]
    return _batch_from_roots(rng, [root], 256, 64, seed, {"name": "tiny"})


def _single_row(make, seed, row_len, name, max_tries=100000):
    for attempt in range(max_tries):
        s = seed + attempt
        rng = np.random.default_rng(s)
        roots = make(rng)
        size = sum(_design_size(r) + _leaves(r) for r in roots)
        if size <= row_len:
            return _batch_from_roots(rng, roots, row_len, 64, s,
                                     {"name": name, "requested_seed": seed,
                                      "design_tokens": size})
    raise RuntimeError(f"{name}: no draw fits {row_len} tokens")


def grpo(seed: int = 1, n_rollouts: int = 16, prefix: int = 5000,
         lo: int = 100, hi: int = 1000, row_len: int = 16384) -> SeqBatch:
    """One GRPO group: non-trainable system prefix + trainable rollouts."""

    def make(rng):
        root = _Node(prefix, False, family=0)
        root.children = [_Node(_uniform(rng, lo, hi), True) for _ in range(n_rollouts)]
        return [root]

    return _single_row(make, seed, row_len, "grpo")


def grpo_tri(seed: int = 1, n_rollouts: int = 16, prefix: int = 5000,
             row_len: int = 16384) -> SeqBatch:
    """Variant of ``grpo`` with rollout lengths 100 + floor(900 B), B ~ Beta(1,2) (mean 400)."""

    def make(rng):
        root = _Node(prefix, False, family=0)
        root.children = [_Node(100 + int(900 * rng.beta(1.0, 2.0)), True)
                         for _ in range(n_rollouts)]
        return [root]

    return _single_row(make, seed, row_len, "grpo_tri")


def curriculum(seed: int = 2, n_families: int = 3, groups_per_family: int = 16,
               completions: int = 8, row_len: int = 4096, system: int = 350,
               instruction: int = 300) -> SeqBatch:
    """System prompt -> task families -> RL groups -> trainable completions.

    Family ids handed to the packer are the RL group index.
    """
    rng = np.random.default_rng(seed)
    root = _Node(system, False)
    g = 0
    for _ in range(n_families):
        fam = _Node(instruction, False)
        for _ in range(groups_per_family):
            grp = _Node(_uniform(rng, 100, 400), False, family=g)
            grp.children = [_Node(_uniform(rng, 50, 300), True) for _ in range(completions)]
            fam.children.append(grp)
            g += 1
        root.children.append(fam)
    return _batch_from_roots(rng, [root], row_len, 64, seed,
                             {"name": "curriculum", "groups": g})


def deep(seed: int = 3, row_len: int = 32768) -> SeqBatch:
    """8192 -> 4 x 2048 -> 4 x U[256,1024] -> 2 x U[64,512] (leaves trainable)."""

    def make(rng):
        root = _Node(8192, False, family=0)
        for _ in range(4):
            b = _Node(2048, False)
            for _ in range(4):
                sb = _Node(_uniform(rng, 256, 1024), False)
                sb.children = [_Node(_uniform(rng, 64, 512), True) for _ in range(2)]
                b.children.append(sb)
            root.children.append(b)
        return [root]

    return _single_row(make, seed, row_len, "deep")


def bushy(seed: int = 4, row_len: int = 16384) -> SeqBatch:
    """1024-token prefix with 512 trainable branches U[8,32], then independent
    trainable sequences U[64,512] while the drawn design still fits the row."""
    rng = np.random.default_rng(seed)
    root = _Node(1024, False, family=0)
    root.children = [_Node(_uniform(rng, 8, 32), True) for _ in range(512)]
    roots = [root]
    used = _design_size(root) + _leaves(root)
    fam = 1
    while True:
        n = _uniform(rng, 64, 512)
        if used + n + 1 > row_len:
            break
        roots.append(_Node(n, True, family=fam))
        used += n + 1
        fam += 1
    return _batch_from_roots(rng, roots, row_len, 64, seed,
                             {"name": "bushy", "design_tokens": used})


def rollout32(seed: int = 0, row_len: int = 131072) -> SeqBatch:
    """The 32-rollout comparison: 4096 root, 12000 group prefix, 8 completions
    per group of 2000 / 2000 / 12000 / 7000 tokens, groups in that order."""
    rng = np.random.default_rng(seed)
    root = _Node(4096, False)
    for g, comp in enumerate((2000, 2000, 12000, 7000)):
        grp = _Node(12000, False, family=g)
        grp.children = [_Node(comp, True) for _ in range(8)]
        root.children.append(grp)
    return _batch_from_roots(rng, [root], row_len, 64, seed, {"name": "rollout32"})


def random_forest(seed: int, n_roots: int = 2, max_depth: int = 3, max_children: int = 3,
                  len_lo: int = 1, len_hi: int = 40, row_len: int = 4096,
                  min_shared: int = 4, trainable_leaves: bool = True,
                  p_nt_leaf: float = 0.2, p_trainable_tail: float = 0.0,
                  vocab: int = VOCAB) -> SeqBatch:
    """Random small forests for property tests.

    Interior nodes are non-trainable; leaves are trainable (or, with
    probability ``p_nt_leaf``, non-trainable).  With ``p_trainable_tail`` a
    non-trainable segment is appended after a trainable leaf (multi-turn
    shape).  A small ``vocab`` provokes accidental token collisions.
    """
    rng = np.random.default_rng(seed)

    def grow(depth):
        n = _Node(_uniform(rng, len_lo, len_hi), False)
        if depth < max_depth and rng.random() < 0.7:
            for _ in range(_uniform(rng, 1, max_children)):
                n.children.append(grow(depth + 1))
        if not n.children:
            n.trainable = trainable_leaves and (rng.random() >= p_nt_leaf)
        return n

    roots = [grow(0) for _ in range(n_roots)]
    firsts: set = set()

    def fill(node, sib):
        toks = rng.integers(0, vocab, size=node.length, dtype=np.int64)
        if vocab >= 64 and node.length > 0:
            while int(toks[0]) in sib:
                toks[0] = rng.integers(0, vocab)
            sib.add(int(toks[0]))
        node.tokens = toks.astype(np.int32)
        s2: set = set()
        for c in node.children:
            fill(c, s2)

    for r in roots:
        fill(r, firsts)
    out = []
    for r in roots:
        _paths(r, [], [], None, out)
    seqs, tr = [], []
    for tok, t, _ in out:
        if p_trainable_tail > 0 and t[-1] == 1 and rng.random() < p_trainable_tail:
            extra = _uniform(rng, 1, 10)
            tok = np.concatenate([tok, rng.integers(0, vocab, extra).astype(np.int32)])
            t = np.concatenate([t, np.zeros(extra, np.uint8)])
        seqs.append(tok.astype(np.int32))
        tr.append(t.astype(np.uint8))
    order = rng.permutation(len(seqs))
    seqs = [seqs[i] for i in order]
    tr = [tr[i] for i in order]
    fam = rng.integers(0, max(1, len(seqs) // 2), size=len(seqs)).astype(np.int32)
    return SeqBatch(seqs, tr, fam, row_len, min_shared, seed, {"name": "random_forest"})


# --------------------------------------------------------------------------
# Attention tensors
# --------------------------------------------------------------------------

@dataclass
class AttnShape:
    n_rows: int
    row_len: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str            # "bf16" or "fp32"
    scale: float
    qkv_std: float = 0.5


CONFIG_SHAPES = {
    "tiny": dict(n_q_heads=1, n_kv_heads=1, head_dim=64, dtype="fp32", qkv_std=1.0),
    "grpo": dict(n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", qkv_std=0.5),
    "curriculum": dict(n_q_heads=16, n_kv_heads=8, head_dim=128, dtype="bf16", qkv_std=0.5),
    "deep": dict(n_q_heads=64, n_kv_heads=8, head_dim=128, dtype="bf16", qkv_std=0.5),
    "bushy": dict(n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", qkv_std=0.5),
}

CONFIG_BATCHES = {"tiny": tiny, "grpo": grpo, "curriculum": curriculum,
                  "deep": deep, "bushy": bushy}
CONFIG_SEEDS = {"tiny": 0, "grpo": 1, "curriculum": 2, "deep": 3, "bushy": 4}


def attn_shape(name: str, n_rows: int, row_len: int) -> AttnShape:
    c = CONFIG_SHAPES[name]
    return AttnShape(n_rows, row_len, c["n_q_heads"], c["n_kv_heads"], c["head_dim"],
                     c["dtype"], 1.0 / float(np.sqrt(c["head_dim"])), c["qkv_std"])


def attn_tensors(shape: AttnShape, seed: int = 0, device="cpu"):
    """Q, K, V [R,T,H,D] and dO [R,T,Hq,D], drawn N(0,1) in fp32 on the CPU
    from a seeded torch generator; Q/K/V scaled by ``qkv_std``; for bf16 the
    values are rounded to bf16 (round-to-nearest-even) and returned as bf16."""
    import torch

    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    R, T, Hq, Hkv, D = (shape.n_rows, shape.row_len, shape.n_q_heads,
                        shape.n_kv_heads, shape.head_dim)
    q = torch.randn(R, T, Hq, D, generator=g, dtype=torch.float32) * shape.qkv_std
    k = torch.randn(R, T, Hkv, D, generator=g, dtype=torch.float32) * shape.qkv_std
    v = torch.randn(R, T, Hkv, D, generator=g, dtype=torch.float32) * shape.qkv_std
    do = torch.randn(R, T, Hq, D, generator=g, dtype=torch.float32)
    if shape.dtype == "bf16":
        q, k, v, do = (t.to(torch.bfloat16) for t in (q, k, v, do))
    return tuple(t.to(device) for t in (q, k, v, do))


def index_tensors(n_rows: int, row_len: int, n_heads: int, head_dim: int, seed: int = 0, device="cpu"):
    """Indexer inputs: q [R, T, H, D] and k [R, T, D] drawn N(0, 1/D) and rounded
    to bf16, w [R, T, H] uniform in [0, 1) float32; seeded CPU torch generator."""
    import torch

    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    s = float(head_dim) ** -0.5
    q = (torch.randn(n_rows, row_len, n_heads, head_dim, generator=g) * s).to(torch.bfloat16)
    k = (torch.randn(n_rows, row_len, head_dim, generator=g) * s).to(torch.bfloat16)
    w = torch.rand(n_rows, row_len, n_heads, generator=g)
    return q.to(device), k.to(device), w.to(device)


def logprob_tensors(n_positions: int, hidden: int, vocab: int, seed: int = 0, logit_std: float = 2.0,
                    device="cpu"):
    """Inputs of the next-token log-probability gather: hidden states h [N, D]
    drawn N(0, 1) and a vocabulary projection W [V, D] drawn N(0, logit_std^2 / D),
    both rounded to bf16 (logits then spread about N(0, logit_std^2)); seeded
    CPU torch generator."""
    import torch

    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    h = torch.randn(n_positions, hidden, generator=g).to(torch.bfloat16)
    w = (torch.randn(vocab, hidden, generator=g) * (logit_std / float(hidden) ** 0.5)).to(torch.bfloat16)
    return h.to(device), w.to(device)


def gdn_tensors(n_tokens: int, n_heads: int, head_dim: int = 128, seed: int = 0, device="cpu"):
    """Gated DeltaNet layer-core inputs: x [N, 3 H d] (the projected q | k | v)
    drawn N(0, 1) and rounded to bf16; conv_w [3 H d, 4] N(0, 1/4) float32;
    g [N, H] = log(U[0.85, 1)) (per-token decays near 1) and beta [N, H] =
    sigmoid(N(0, 1)), float32; seeded CPU torch generator."""
    import torch

    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    C = 3 * n_heads * head_dim
    x = torch.randn(n_tokens, C, generator=gen).to(torch.bfloat16)
    conv_w = torch.randn(C, 4, generator=gen) * 0.5
    g = torch.log(0.85 + 0.15 * torch.rand(n_tokens, n_heads, generator=gen))
    beta = torch.sigmoid(torch.randn(n_tokens, n_heads, generator=gen))
    return tuple(t.to(device) for t in (x, conv_w, g, beta))
