"""Oracle: prefix-tree construction, tree-aware bin packing, materialization.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (prefix-tree-packing page, furtherai.github.io):
  * tree build section -- the recursive walk: emit the longest run every
    active sequence agrees on once, split the rest by next token, recurse;
    sequences no longer than the current start drop out.
  * "Two refinements" -- a minimum shared-segment length (default 64) and
    no sharing of trainable tokens.
  * "an off-by-one note" -- each branch keeps one duplicated, non-trainable
    context token at its join point so it has its own query for the first
    unique token.  The 32-rollout section fixes where it applies: the
    accounting is "11,999 shared group-prefix tokens plus completion-length
    + 1 tokens per rollout" while the 4096-token root is paid in full, i.e.
    the copy is made only where a member's next token is trainable.
  * "A simple boundary ..." -- one global tree over every queued sequence.
  * bin packing section -- a bin holds leaves, the set of occupied segments
    and a token count; a leaf's insertion delta is the summed length of its
    path segments the bin does not hold yet; groups are ordered by their most
    expensive leaf (descending); each leaf goes to the feasible bin with the
    least room left (strict improvement, so the earliest bin wins ties), a
    new bin only when none fits.
  * "You can also just fill in the bins as you go" / the 32-rollout table --
    the in-order placement used as the comparison arm.
  * materialization section -- the plan is integers only; tokens are sliced
    into rows in one pass.
  * attention section -- a DFS assigns increasing indices and every token
    has an [enter, exit] interval; ``subtree_end`` is the exit index.

Readings where the pages are silent:
  * the minimum length is tested on the agreed run, before the join copy is
    carved out of it;
  * a run shorter than the minimum is not emitted but pushed down into every
    sub-partition, so a deeper long run can still be shared;
  * children and roots are ordered by (token at the split, or -1 when the
    sequence ended there; then the smallest member index);
  * a group for placement is the caller's family id; without family ids each
    sequence is its own family;
  * rows hold the DFS pre-order of the bin's segments, padded at the end with
    token 0, position 0, subtree_end = own index, loss 0;
  * position id = index of the token in its original sequence;
  * loss_mask[x] = 1 iff the next token of x's sequence is trainable.
"""
from __future__ import annotations

import sys
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np


class PackError(ValueError):
    """Raised for inputs the packer rejects (mirrors the C status codes)."""

    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


@dataclass
class Segment:
    sid: int
    parent: int          # -1 for a root
    lo: int              # first covered position in every member sequence
    hi: int              # one past the last covered position
    rep: int             # index of a member sequence (token source)
    is_leaf: bool = False

    @property
    def length(self) -> int:
        return self.hi - self.lo


@dataclass
class Trie:
    segments: List[Segment]
    leaf_of: List[int]                   # sequence -> its leaf segment id
    seqs: List[np.ndarray]
    trainable: List[np.ndarray]

    def path(self, s: int) -> List[int]:
        """Segment ids on sequence s's root-to-leaf path."""
        out = []
        x = self.leaf_of[s]
        while x >= 0:
            out.append(x)
            x = self.segments[x].parent
        return out[::-1]


def leading_nontrainable(tr: np.ndarray) -> int:
    """Number of leading non-trainable tokens of a sequence."""
    idx = np.flatnonzero(np.asarray(tr) != 0)
    return int(idx[0]) if idx.size else int(len(tr))


def build_trie(seqs: Sequence[np.ndarray], trainable: Sequence[np.ndarray],
               min_shared: int = 64, groups: Optional[List[List[int]]] = None) -> Trie:
    """Walk all sequences into one prefix forest (or one per group).

    ``groups`` lists sequence indices per independent tree (the per-group
    comparison arm); by default all sequences form one global forest.
    """
    n = len(seqs)
    seqs = [np.asarray(s, dtype=np.int64) for s in seqs]
    trainable = [np.asarray(t, dtype=np.uint8) for t in trainable]
    L = [len(s) for s in seqs]
    nt = [leading_nontrainable(t) for t in trainable]
    for s in range(n):
        if L[s] == 0:
            raise PackError("EINVAL", f"sequence {s} is empty")
    segs: List[Segment] = []
    leaf_of = [-1] * n

    def emit(parent, lo, hi, rep, leaf=False):
        segs.append(Segment(len(segs), parent, lo, hi, rep, leaf))
        return len(segs) - 1

    def agreed_run(S, start):
        # largest a: every member is non-trainable on [start, start+a) and
        # all members carry the same tokens there
        lim = min(nt[s] for s in S) - start
        if lim <= 0:
            return 0
        first = seqs[S[0]][start:start + lim]
        a = lim
        for s in S[1:]:
            diff = np.flatnonzero(seqs[s][start:start + lim] != first)
            if diff.size:
                a = min(a, int(diff[0]))
        return a

    def partition(S, p):
        parts = []
        by_tok: Dict[int, List[int]] = {}
        for s in S:
            if L[s] == p:
                parts.append(((-1, s), [s]))
            elif trainable[s][p]:
                parts.append(((int(seqs[s][p]), s), [s]))
            else:
                by_tok.setdefault(int(seqs[s][p]), []).append(s)
        for tok, members in by_tok.items():
            parts.append(((tok, min(members)), members))
        parts.sort(key=lambda x: x[0])
        return [m for _, m in parts]

    def build(S, start, parent):
        if len(S) == 1:
            s = S[0]
            leaf_of[s] = emit(parent, start, L[s], s, leaf=True)
            return
        A = agreed_run(S, start)
        if A >= min_shared:
            E = start + A
            join = any(nt[s] == E and E < L[s] for s in S)
            seg_end = E - 1 if join else E
            node = parent
            if seg_end > start:
                node = emit(parent, start, seg_end, S[0])
            for part in partition(S, E):
                build(part, seg_end, node)
        else:
            for part in partition(S, start + A):
                build(part, start, parent)

    old = sys.getrecursionlimit()
    sys.setrecursionlimit(max(old, 100000))
    try:
        for G in (groups if groups is not None else [list(range(n))]):
            if G:
                build(sorted(G), 0, -1)
    finally:
        sys.setrecursionlimit(old)
    return Trie(segs, leaf_of, seqs, trainable)


# ---------------------------------------------------------------------------
# Bin packing
# ---------------------------------------------------------------------------

@dataclass
class Leaf:
    seq: int
    segment_path: List[tuple]            # [(segment id, length)] root -> leaf
    empty_bin_cost: int


@dataclass
class Bin:
    leaves: List[Leaf] = field(default_factory=list)
    occupied: set = field(default_factory=set)
    token_count: int = 0

    def insertion_delta(self, leaf: Leaf) -> int:
        return sum(ln for sid, ln in leaf.segment_path if sid not in self.occupied)

    def add(self, leaf: Leaf) -> None:
        self.token_count += self.insertion_delta(leaf)
        self.occupied.update(sid for sid, _ in leaf.segment_path)
        self.leaves.append(leaf)


def make_leaves(trie: Trie) -> List[Leaf]:
    out = []
    for s in range(len(trie.seqs)):
        path = [(sid, trie.segments[sid].length) for sid in trie.path(s)]
        # every position of the sequence lies on exactly one path segment, so
        # the full unshared cost is the sequence length
        out.append(Leaf(s, path, int(sum(ln for _, ln in path))))
    return out


def family_groups(n: int, family: Optional[Sequence[int]]) -> List[List[int]]:
    """Sequence indices per family, families in order of first appearance."""
    if family is None:
        return [[s] for s in range(n)]
    order: Dict[int, List[int]] = {}
    for s in range(n):
        order.setdefault(int(family[s]), []).append(s)
    return list(order.values())


def place_bfd(leaves: List[Leaf], groups: List[List[int]], row_len: int) -> List[Bin]:
    """Tree-aware best-fit-decreasing over groups of leaves."""
    for lf in leaves:
        if lf.empty_bin_cost > row_len:
            raise PackError("ETOOLONG", f"sequence {lf.seq} has {lf.empty_bin_cost} > {row_len}")
    glv = [[leaves[s] for s in g] for g in groups]
    # Python's sort is stable, also with reverse=True
    ordered = sorted(glv, key=lambda g: max(lf.empty_bin_cost for lf in g), reverse=True)
    bins: List[Bin] = []
    for g in ordered:
        for lf in g:
            best, best_room = None, row_len + 1
            for b in bins:
                count = b.token_count + b.insertion_delta(lf)
                if count <= row_len and row_len - count < best_room:
                    best, best_room = b, row_len - count
            if best is None:
                best = Bin()
                bins.append(best)
            best.add(lf)
    return bins


def place_in_order(leaves: List[Leaf], row_len: int) -> List[Bin]:
    """Fill one row at a time in input order; move on when a leaf does not fit."""
    bins: List[Bin] = []
    for lf in leaves:
        if lf.empty_bin_cost > row_len:
            raise PackError("ETOOLONG", f"sequence {lf.seq}")
        if not bins or bins[-1].token_count + bins[-1].insertion_delta(lf) > row_len:
            bins.append(Bin())
        bins[-1].add(lf)
    return bins


# ---------------------------------------------------------------------------
# Materialization
# ---------------------------------------------------------------------------

@dataclass
class RowSeg:
    sid: int
    parent: int          # parent segment id (-1 root)
    row_start: int       # first row index of the segment
    length: int
    lo: int              # first sequence position covered


@dataclass
class Plan:
    row_len: int
    token_ids: np.ndarray        # int32 [R, T]
    position_ids: np.ndarray     # int32 [R, T]
    subtree_end: np.ndarray      # int32 [R, T]
    loss_mask: np.ndarray        # uint8 [R, T]
    gather_index: np.ndarray     # int64 [sum len]
    used: List[int]              # real tokens per row
    row_segments: List[List[RowSeg]]
    trie: Trie
    bins: List[Bin]

    @property
    def n_rows(self) -> int:
        return len(self.bins)


def materialize(trie: Trie, bins: List[Bin], row_len: int) -> Plan:
    R, T = len(bins), row_len
    tok = np.zeros((R, T), np.int32)
    pos = np.zeros((R, T), np.int32)
    se = np.zeros((R, T), np.int32)
    lm = np.zeros((R, T), np.uint8)
    offs = np.zeros(len(trie.seqs) + 1, np.int64)
    offs[1:] = np.cumsum([len(s) for s in trie.seqs])
    gather = np.full(int(offs[-1]), -1, np.int64)
    used, row_segs = [], []
    for r, b in enumerate(bins):
        # segment ids are handed out as the walk emits them, parents first and
        # each subtree contiguously, so ascending id order is a DFS pre-order
        occ = sorted(b.occupied)
        start: Dict[int, int] = {}
        cur = 0
        rs = []
        for sid in occ:
            sg = trie.segments[sid]
            start[sid] = cur
            rs.append(RowSeg(sid, sg.parent, cur, sg.length, sg.lo))
            src = trie.seqs[sg.rep]
            tok[r, cur:cur + sg.length] = src[sg.lo:sg.hi]
            pos[r, cur:cur + sg.length] = np.arange(sg.lo, sg.hi)
            cur += sg.length
        assert cur == b.token_count <= T
        # exit index: the last row index of any occupied descendant-or-self
        occset = set(occ)
        last = {sid: (start[sid] + trie.segments[sid].length - 1) for sid in occ}
        for sid in occ:
            if trie.segments[sid].length == 0:
                continue
            end = start[sid] + trie.segments[sid].length - 1
            x = trie.segments[sid].parent
            while x >= 0:
                assert x in occset
                last[x] = max(last[x], end)
                x = trie.segments[x].parent
        for sid in occ:
            n = trie.segments[sid].length
            se[r, start[sid]:start[sid] + n] = last[sid]
        for j in range(cur, T):            # pads
            se[r, j] = j
        for lf in b.leaves:
            s = lf.seq
            tr = trie.trainable[s]
            for sid, _ in lf.segment_path:
                sg = trie.segments[sid]
                n = sg.length
                xs = start[sid] + np.arange(n)
                gather[offs[s] + sg.lo: offs[s] + sg.hi] = r * T + xs
                # loss at x <=> the token after x in this sequence is trainable
                nxt = np.zeros(n, np.uint8)
                m = min(sg.hi + 1, len(tr)) - (sg.lo + 1)
                if m > 0:
                    nxt[:m] = tr[sg.lo + 1: sg.lo + 1 + m]
                lm[r, xs] = np.maximum(lm[r, xs], nxt)
        used.append(cur)
        row_segs.append(rs)
    assert (gather >= 0).all()
    return Plan(T, tok, pos, se, lm, gather, used, row_segs, trie, bins)


def pack(seqs, trainable, row_len: int, min_shared: int = 64, family=None,
         per_family: bool = False, in_order: bool = False) -> Plan:
    """Whole planning + materialization pass.

    ``per_family`` builds one tree per family before packing (the
    "tree per RL group" comparison arm); ``in_order`` uses the in-order
    placement instead of best-fit-decreasing.
    """
    if row_len <= 0 or min_shared < 1:
        raise PackError("EINVAL", "row_len must be > 0 and min_shared >= 1")
    n = len(seqs)
    groups = family_groups(n, family)
    trie = build_trie(seqs, trainable, min_shared, groups if per_family else None)
    leaves = make_leaves(trie)
    if in_order:
        bins = place_in_order(leaves, row_len)
    else:
        bins = place_bfd(leaves, groups, row_len)
    return materialize(trie, bins, row_len)


def plan_info(plan: Plan) -> dict:
    inp = int(sum(len(s) for s in plan.trie.seqs))
    packed = int(sum(plan.used))
    return {
        "n_rows": plan.n_rows,
        "row_len": plan.row_len,
        "input_tokens": inp,
        "packed_tokens": packed,
        "n_segments": len(plan.trie.segments),
        "n_leaves": len(plan.trie.seqs),
        "tree_token_ratio": (inp / packed) if packed else 0.0,
    }
