"""Benchmark of the prefix-tree tree-attention path on GB300.

One step = the whole path over one batch: host packing (trie walk, tree-aware
best-fit-decreasing, materialization) -> copy of the row metadata to the GPU
-> tile classification -> forward (O, LSE) -> backward (dQ, dK, dV).
As a data loader would, the host packs the next step's batch while the GPU
runs the current step (two pinned metadata sets); a step's time is the GPU
time from its metadata upload to the end of its backward, and the host pack
time is reported beside it.  Q, K, V and dO are resident in HBM when the
timed region starts; L2 is flushed (a 512 MiB write on the GPU, outside the
step's events) before every timed step.  The end-to-end leg does the same
through the host-buffer call (inputs uploaded, outputs downloaded per step).

Metric: useful tree-attention fwd+bwd TFLOP/s, where useful work counts each
visible (query, key) pair once per query head: 4 * D flops forward and
10 * D backward (the FlashAttention convention, recomputation of S included);
masked or skipped work is not counted.  Trajectories/s = sequences per step
/ step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank packs and processes its own batch
(weak scaling, no collective on the data path); the step time is the maximum
over ranks.  --impl reference times the CPU oracle (float64 NumPy) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sft_trie_build_gb300 import workloads as W  # noqa: E402
from sft_trie_build_gb300.shard import max_over_ranks, rank_seed  # noqa: E402

WORKLOAD = "grpo"
WORKLOAD_DESC = ("one GRPO group: 5000-token non-trainable system prefix + 16 trainable rollouts "
                 "U[100,1000], packed into one 16384-token row; bf16 attention, 32 query heads, "
                 "8 kv heads, head_dim 128, scale 1/sqrt(128)")
METRIC = "tree-attn fwd+bwd useful TFLOP/s (% of BF16 peak) and trajectories/s on 1 GB300"


# DRAM bytes (read + write) of one backward call on the workload above, from
# one ncu capture of every launch of the second call of
#   python bench.py --profile attn --reps 1
# (dram__bytes_read.sum + dram__bytes_write.sum, -s 22 -c 22): bwd_delta_kernel
# 270.6e6 + 22.6e6, the eight bwd_tc_kernel launches 617.5e6 + 3677.4e6, the
# eight dq_tc_kernel launches 4152.3e6 + 53.1e6.  To be retaken whenever one of
# the three kernels changes.
BWD_DRAM_BYTES = 270577152 + 22558976 + 617461504 + 3677415936 + 4152305920 + 53067264


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


def _indexer(R, T, se, tile_meta, pairs, useful, dev, heads=8, dim=64, top_k=512, reps=10) -> dict:
    """The tree-aware top-k indexer on the same packed row (device leg's
    classification): scoring over ancestor candidates + top-k selection."""
    import torch
    from sft_trie_build_gb300 import stp

    q, k, w = (x.to(dev) for x in W.index_tensors(R, T, heads, dim, seed=23))
    idesc = stp.index_desc(R, T, heads, dim, top_k, pairs)
    ws = torch.empty(stp.stp_index_workspace_size(idesc), dtype=torch.uint8, device=dev)
    idx = torch.empty(R, T, top_k, dtype=torch.int32, device=dev)
    sc = torch.empty(R, T, top_k, dtype=torch.float32, device=dev)
    for _ in range(3):
        stp.stp_index_topk(idesc, q, k, w, se, tile_meta, idx, sc, ws)
    torch.cuda.synchronize()
    assert stp.stp_device_status(ws) == stp.STP_OK
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        stp.stp_index_topk(idesc, q, k, w, se, tile_meta, idx, sc, ws)
    e.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / reps
    return {"heads": heads, "head_dim": dim, "top_k": top_k, "ms": ms,
            "candidate_pairs_per_s": useful / (ms / 1e3),
            "useful_scoring_tflops": 2.0 * heads * dim * useful / (ms / 1e3) / 1e12}


def _logprob(tok, mask, dev, peak, hidden=4096, vocab=151936, reps=10) -> dict:
    """Next-token log-probabilities of the packed row's loss positions (its
    loss mask and targets from the packer) under a synthetic vocabulary
    projection: stp_logprob_gather (tiles list + tcgen05 logits with an online
    log-sum-exp + split combine).  W alone (1.2 GB) exceeds L2."""
    import torch
    from sft_trie_build_gb300 import stp

    R, T = tok.shape
    h, w = (x.to(dev) for x in W.logprob_tensors(R * T, hidden, vocab, seed=29))
    tok_d = torch.from_numpy(np.ascontiguousarray(tok)).to(dev)
    mask_d = torch.from_numpy(np.ascontiguousarray(mask)).to(dev)
    desc = stp.logprob_desc(R, T, hidden, vocab)
    ws = torch.empty(stp.stp_logprob_workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty(R * T, dtype=torch.float32, device=dev)
    for _ in range(3):
        stp.stp_logprob_gather(desc, h, w, tok_d, mask_d, out, ws)
    torch.cuda.synchronize()
    assert stp.stp_device_status(ws) == stp.STP_OK
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        stp.stp_logprob_gather(desc, h, w, tok_d, mask_d, out, ws)
    e.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / reps
    m = np.asarray(mask).reshape(-1) != 0
    n_loss = int(m.sum())
    tiles = int(len(np.unique(np.flatnonzero(m) // 128)))
    useful = 2.0 * n_loss * vocab * hidden / (ms / 1e3) / 1e12
    computed = 2.0 * tiles * 128 * vocab * hidden / (ms / 1e3) / 1e12
    return {"hidden": hidden, "vocab": vocab, "loss_positions": n_loss, "tiles_with_loss": tiles, "ms": ms,
            "useful_tflops": useful, "computed_tflops": computed, "frac_of_bf16_peak": useful / peak,
            "launches_per_call": 3}


def _gdn(meta, dev, heads=16, reps=10) -> dict:
    """Tree-aware Gated DeltaNet layer core over the packed row, 16 heads of
    128: the forward (path convolution, per-chunk prep, one state pass per
    tree depth; stp_gdn_fwd), then the training forward (stp_gdn_fwd_train)
    and the backward (stp_gdn_bwd)."""
    import torch
    from sft_trie_build_gb300 import stp

    se = meta["subtree_end"]
    R, T = se.shape
    # real tokens per row: one past the last row position any sequence occupies (pads follow)
    gi = np.asarray(meta["gather_index"])
    used = np.zeros(R, np.int64)
    np.maximum.at(used, gi // T, gi % T + 1)
    desc = stp.gdn_desc(R, T, heads)
    t0 = time.perf_counter()
    plan = stp.stp_gdn_plan(desc, se, used.astype(np.int32))
    plan_ms = 1e3 * (time.perf_counter() - t0)
    d_plan = torch.from_numpy(plan).to(dev)
    x, cw, g, beta = (t.to(dev) for t in W.gdn_tensors(R * T, heads, 128, seed=31))
    ws = torch.empty(stp.stp_gdn_workspace_size(desc, plan), dtype=torch.uint8, device=dev)
    o = torch.empty(R * T, heads, 128, dtype=torch.float32, device=dev)
    for _ in range(3):
        stp.stp_gdn_fwd(desc, plan, d_plan, x, cw, g, beta, o, ws)
    torch.cuda.synchronize()
    assert stp.stp_device_status(ws) == stp.STP_OK
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        stp.stp_gdn_fwd(desc, plan, d_plan, x, cw, g, beta, o, ws)
    e.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / reps
    real = int(used.sum())
    out = {"heads": heads, "head_dim": 128, "tokens": real, "segments": int(plan[stp.GP_NSEG]),
           "chunks": int(plan[stp.GP_NCHUNK]), "depths": int(plan[stp.GP_NDEPTH]), "ms": ms,
           "tokens_per_s": real / (ms / 1e3), "host_plan_ms": plan_ms,
           # convolution, the preparation (depth 0, depth 1 and the deeper depths apart), a walk per depth
           "launches_per_call": 1 + min(int(plan[stp.GP_NDEPTH]), 3) + int(plan[stp.GP_NDEPTH])}
    # training: the forward that keeps the chunk states, then the backward
    try:
        tws = torch.empty(stp.stp_gdn_train_workspace_size(desc, plan), dtype=torch.uint8, device=dev)
        d_o = torch.randn(R * T, heads, 128, device=dev)
        dx = torch.empty(R * T, 3 * heads * 128, device=dev)
        dw = torch.empty(3 * heads * 128, 4, device=dev)
        dg = torch.empty(R * T, heads, device=dev)
        db = torch.empty(R * T, heads, device=dev)
        legs = {"fwd_train": lambda: stp.stp_gdn_fwd_train(desc, plan, d_plan, x, cw, g, beta, o, tws),
                "bwd": lambda: stp.stp_gdn_bwd(desc, plan, d_plan, x, cw, g, beta, d_o, dx, dw, dg, db, tws)}
        for _ in range(2):
            legs["fwd_train"]()
            legs["bwd"]()
        torch.cuda.synchronize()
        for name, fn in legs.items():
            a.record()
            for _ in range(3):
                fn()
            e.record()
            torch.cuda.synchronize()
            out[name + "_ms"] = a.elapsed_time(e) / 3
        out["train_status"] = stp.stp_device_status(tws)
    except Exception as exc:   # an auxiliary field: report, do not lose the bench line
        out["train_error"] = repr(exc)
    return out


def _what_if(n_candidates: int = 64, groups_per_candidate: int = 8) -> dict:
    """Host 'what if' planning: rows that candidate batches (whole groups drawn
    from the curriculum pool) would need, global tree vs one tree per group,
    planned in parallel without materializing anything."""
    from sft_trie_build_gb300 import stp

    b = W.curriculum(W.CONFIG_SEEDS["curriculum"])
    tokens, offsets, train = b.flat()
    fam = np.asarray(b.family)
    groups = np.unique(fam)
    rng = np.random.default_rng(11)
    subsets = [np.flatnonzero(np.isin(fam, rng.choice(groups, groups_per_candidate, replace=False)))
               for _ in range(n_candidates)]
    kw = dict(row_len=b.row_len, min_shared=b.min_shared)
    stp.stp_plan_rows_many(tokens, offsets, train, b.family, subsets[:2], **kw)  # warm-up
    t0 = time.perf_counter()
    rows, _ = stp.stp_plan_rows_many(tokens, offsets, train, b.family, subsets, **kw)
    dt = time.perf_counter() - t0
    rows_pf, _ = stp.stp_plan_rows_many(tokens, offsets, train, b.family, subsets, flags=stp.STP_PER_FAMILY, **kw)
    return {"pool": f"curriculum config: {len(b.seqs)} sequences in {len(groups)} groups, rows of {b.row_len}",
            "candidates": n_candidates, "groups_per_candidate": groups_per_candidate,
            "ms_total": 1e3 * dt, "ms_per_candidate": 1e3 * dt / n_candidates,
            "host_threads": os.cpu_count(), "rows_mean_global_tree": float(np.mean(rows)),
            "rows_mean_tree_per_group": float(np.mean(rows_pf))}


def _time_batch(b, name, dev, flush, reps=10, min_shared=None, seed=41):
    """Packs batch `b` (stp_pack, optionally with another minimum shared run)
    and times classification, forward and backward (forward only for the
    float32 path) with CUDA events, L2 flushed before every repetition
    (median of `reps`).  Returns (timings dict, plan info, host inputs)."""
    import torch
    from sft_trie_build_gb300 import stp

    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len,
                        min_shared=b.min_shared if min_shared is None else min_shared)
    info = stp.stp_plan_info(plan)
    meta = stp.stp_plan_write(plan)
    R, T = info["n_rows"], b.row_len
    shape = W.attn_shape(name, R, T)
    Hq, Hkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    bf16 = shape.dtype == "bf16"
    host = W.attn_tensors(shape, seed)
    q, k, v, do = (x.to(dev) for x in host)
    se_np = meta["subtree_end"]
    pairs = stp.stp_count_tile_pairs(se_np)
    # dS tiles of two kv-head groups at a time where all groups' would pass 8 GB
    ds_groups = 2 if bf16 and pairs * Hq * 32768 > 8e9 else 0
    desc = stp.Desc(R, T, Hq, Hkv, D, stp.STP_BF16 if bf16 else stp.STP_FP32, shape.scale, pairs,
                    ds_groups=ds_groups)
    buf = stp.Buffers(desc, dev)
    ws_bytes = sum(stp.stp_workspace_size(desc))
    se = torch.from_numpy(se_np).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(R, Hq, T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def once(m=None):
        if m:
            m[0].record()
        stp.stp_classify(desc, se, buf.tile_meta)
        if m:
            m[1].record()
        stp.stp_attn_fwd(desc, q, k, v, se, buf.tile_meta, o, lse, buf.fwd_ws)
        if m:
            m[2].record()
        if bf16:
            stp.stp_attn_bwd(desc, q, k, v, o, lse, do, se, buf.tile_meta, dq, dk, dv, buf.bwd_ws)
        if m:
            m[3].record()

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    marks = []
    for _ in range(reps):
        flush.fill_(1)
        m = (ev(), ev(), ev(), ev())
        once(m)
        marks.append(m)
    torch.cuda.synchronize()
    for ws in (buf.tile_meta, buf.fwd_ws) + ((buf.bwd_ws,) if bf16 else ()):
        assert stp.stp_device_status(ws) == stp.STP_OK
    t = {"classify_ms": statistics.median(a.elapsed_time(c) for a, c, _, _ in marks),
         "fwd_ms": statistics.median(c.elapsed_time(f) for _, c, f, _ in marks),
         "bwd_ms": statistics.median(f.elapsed_time(e) for _, _, f, e in marks) if bf16 else 0.0,
         "ms": statistics.median(a.elapsed_time(e) for a, _, _, e in marks),
         "tile_pairs": int(desc.max_tile_pairs), "shape": shape, "bf16": bf16,
         "ds_groups_held": ds_groups or min(Hkv, 8), "device_workspace_gb": ws_bytes / 1e9}
    del buf, q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    return t, info, host


def _attn_config(name, dev, peak, flush, reps=10, oracle_heads=1) -> dict:
    """One of the other workloads through the same calls (classification,
    forward, backward; forward only for the float32 tiny row), with beside it
    the float64 oracle on `oracle_heads` query heads of the same packed batch
    (a bounded sample of the same work)."""
    b = W.CONFIG_BATCHES[name](W.CONFIG_SEEDS[name])
    t, info, host = _time_batch(b, name, dev, flush, reps)
    shape, bf16 = t["shape"], t["bf16"]
    R, T = info["n_rows"], b.row_len
    Hq, Hkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    useful = float(info["useful_pairs"])
    flops = (14.0 if bf16 else 4.0) * D * Hq * useful
    tot = t["ms"]
    nt = T // 128
    out = {"workload": b.info.get("name", name), "rows": R, "row_len": T, "sequences": b.n_seqs,
           "heads": f"{Hq}/{Hkv}", "head_dim": D, "dtype": shape.dtype,
           "passes": "classify+fwd+bwd" if bf16 else "classify+fwd",
           "input_tokens": info["input_tokens"], "packed_tokens": info["packed_tokens"],
           "useful_pairs_per_head": int(useful), "tile_pairs": t["tile_pairs"],
           "tile_grid": f"{R} x {nt} x {nt}",
           "classify_ms": t["classify_ms"], "fwd_ms": t["fwd_ms"], "bwd_ms": t["bwd_ms"], "ms": tot,
           "useful_tflops": flops / (tot / 1e3) / 1e12,
           "trajectories_per_s": b.n_seqs / (tot / 1e3),
           "packed_tokens_per_s": info["packed_tokens"] / (tot / 1e3),
           "l2": "flushed (512 MiB write) before every repetition; median of %d" % reps,
           "ds_groups_held": t["ds_groups_held"], "device_workspace_gb": t["device_workspace_gb"]}
    if bf16:
        out["pct_of_bf16_peak"] = 100.0 * out["useful_tflops"] / peak
        out["fwd_tflops"] = 4.0 * D * Hq * useful / (t["fwd_ms"] / 1e3) / 1e12
        out["bwd_tflops"] = 10.0 * D * Hq * useful / (t["bwd_ms"] / 1e3) / 1e12
    if oracle_heads:
        from oracle import attn as OA
        from oracle import pack as OP
        plan_o = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
        q_h, k_h, v_h, do_h = (x.float() for x in host)
        if bf16:
            dt, fl = oracle_sample(plan_o, q_h, k_h, v_h, do_h, shape.scale, oracle_heads)
        else:
            t0 = time.perf_counter()
            OA.attn_fwd(plan_o, q_h[:, :, :oracle_heads], k_h[:, :, :1], v_h[:, :, :1], shape.scale)
            dt = time.perf_counter() - t0
            fl = 4.0 * D * oracle_heads * OA.useful_pairs(plan_o)
        out["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                               "kind": "oracle", "seconds": dt,
                               "sample": f"float64 NumPy oracle, {'fwd+bwd' if bf16 else 'fwd'} of "
                                         f"{oracle_heads} of {Hq} query heads over the whole packed batch"}
    return out


def _list_mode(dev, peak, flush, reps=10) -> dict:
    """The GRPO batch packed as a tree and without sharing ("list mode":
    every sequence its own root, no shared run being long enough), rows of the
    same length, through the same calls and timing (classification, forward,
    backward); the pair token-throughput change / trajectory-throughput ratio
    (attention only) sits beside the CoreWeave page's end-to-end 6.8x / -15%."""
    b = _batch()
    tree, tinfo, _ = _time_batch(b, WORKLOAD, dev, flush, reps, seed=43)
    lst, linfo, _ = _time_batch(b, WORKLOAD, dev, flush, reps, min_shared=1 << 30, seed=43)
    shape = lst["shape"]
    D, Hq = shape.head_dim, shape.n_q_heads

    def leg(t, info):
        ms = t["ms"]
        fl = 14.0 * D * Hq * float(info["useful_pairs"])
        return {"rows": info["n_rows"], "packed_tokens": info["packed_tokens"],
                "useful_pairs_per_head": int(info["useful_pairs"]), "ms": ms,
                "useful_tflops": fl / (ms / 1e3) / 1e12,
                "pct_of_bf16_peak": 100.0 * fl / (ms / 1e3) / 1e12 / peak,
                "trajectories_per_s": b.n_seqs / (ms / 1e3),
                "packed_tokens_per_s": info["packed_tokens"] / (ms / 1e3)}

    lt, ll = leg(tree, tinfo), leg(lst, linfo)
    return {"workload": f"the GRPO batch ({b.n_seqs} sequences of 5000 + U[100,1000] tokens), rows of "
                        f"{b.row_len}: prefix tree vs list mode (no sharing: each sequence its own root)",
            "tree": lt, "list": ll,
            "token_throughput_change": lt["packed_tokens_per_s"] / ll["packed_tokens_per_s"] - 1.0,
            "trajectory_throughput_ratio": lt["trajectories_per_s"] / ll["trajectories_per_s"],
            "token_density": ll["packed_tokens"] / lt["packed_tokens"],
            "pages_context": "CoreWeave ART-Optimized Megatron page: 6.8x trajectories/s at -15% tokens/s "
                             "(end-to-end training step, GPU not named); ~8x theoretical bound"}


def _planning_cost(reps=3) -> dict:
    """Host planning cost of the packer (stp_pack: trie walk and placement
    timed apart inside the call; stp_plan_write timed around the call) on the
    global-tree curriculum batch at 1/4, 1, 4 and 16 times its 48 groups,
    beside the prefix-tree-packing page's planning-cost table (a Python
    implementation on unnamed hardware)."""
    from sft_trie_build_gb300 import stp

    page = {12: (105, 0.9, 1.4, 15), 48: (450, 9.6, 4.2, 61), 192: (1668, 42.0, 48.7, 227),
            768: (6686, 291.2, 743.5, 918)}
    out = []
    for gpf in (4, 16, 64, 256):
        b = W.curriculum(W.CONFIG_SEEDS["curriculum"], groups_per_family=gpf)
        tokens, offsets, train = b.flat()
        runs = []
        for _ in range(reps):
            t0 = time.perf_counter()
            plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=b.min_shared)
            t1 = time.perf_counter()
            stp.stp_plan_write(plan)
            t2 = time.perf_counter()
            tm = stp.stp_plan_times(plan)
            runs.append((tm["walk_ms"], tm["place_ms"], 1e3 * (t1 - t0), 1e3 * (t2 - t1)))
        walk, place, pack, write = (statistics.median(r[i] for r in runs) for i in range(4))
        groups = 3 * gpf
        info = stp.stp_plan_info(plan)
        row = {"groups": groups, "completions": b.n_seqs, "input_tokens": info["input_tokens"],
               "rows": info["n_rows"], "tree_walk_ms": walk, "placement_ms": place, "stp_pack_ms": pack,
               "materialize_ms": write}
        if groups in page:
            c, pw, pb, pr = page[groups]
            row["page"] = {"completions": c, "tree_walk_ms": pw, "bin_packing_ms": pb, "rows": pr}
        out.append(row)
    return {"rows_of": "rows of 4096 tokens, min shared run 64, one global tree, host C++ packer, one thread",
            "median_of": reps, "batches": out}


def _classify_bandwidth(desc, se, tile_meta, reps=20) -> dict:
    """Tile classification (three kernels) timed alone on the benchmarked row,
    against its algorithmic bytes: subtree_end read once (4 B per token), the
    class matrix written (1 B per tile pair), and per non-empty pair the two
    list entries, the rank and the pair index (16 B)."""
    import torch
    from sft_trie_build_gb300 import stp

    for _ in range(3):
        stp.stp_classify(desc, se, tile_meta)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        stp.stp_classify(desc, se, tile_meta)
    e.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / reps
    R, T = desc.n_rows, desc.row_len
    nt = T // 128
    by = 4 * R * T + R * nt * nt + 16 * int(desc.max_tile_pairs)
    return {"kernels": "tile_minmax_kernel + tile_lists_kernel + tile_pairs_kernel + tile_pair_index_kernel", "ms": ms,
            "algorithmic_bytes": by, "achieved_gbs": by / (ms / 1e3) / 1e9,
            "bound": "latency (the whole row's metadata is ~0.3 MB; back-to-back launches, L2-resident)"}


def _batch(rank=0):
    return W.grpo(rank_seed(W.CONFIG_SEEDS[WORKLOAD], rank))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms; `stop(t0, t1)`
    keeps the samples taken between two host wall-clock times (the timed
    region) and summarizes those."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0=None, t1=None):
        import datetime

        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sms, mx, reasons, power, total = [], None, set(), [], 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smx, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            total += 1
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            sms.append(sm)
            mx = smx
            power.append(pw)
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms), "samples_total": total,
                "power_w_max": max(power) if power else None,
                "window": "samples taken inside the timed region (every 50 ms)"}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


def oracle_sample(plan_o, q, k, v, do, scale, heads=1):
    """Float64 oracle fwd+bwd on the first `heads` query heads (and the kv
    heads they read); returns (seconds, useful flops of the sample)."""
    from oracle import attn as OA
    G = q.shape[2] // k.shape[2]
    nkv = -(-heads // G)
    qs, ks, vs, dos = q[:, :, :heads], k[:, :, :nkv], v[:, :, :nkv], do[:, :, :heads]
    pairs = OA.useful_pairs(plan_o)
    t0 = time.perf_counter()
    OA.attn_bwd(plan_o, qs, ks, vs, dos, scale)
    dt = time.perf_counter() - t0
    return dt, 14.0 * q.shape[-1] * heads * pairs


def run_reference(args, rank, world):
    """The CPU oracle timed on this host's cores, a bounded sample per step."""
    if rank != 0:
        return
    from oracle import pack as OP
    b = _batch()
    plan_o = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
    shape = W.attn_shape(WORKLOAD, plan_o.n_rows, b.row_len)
    q, k, v, do = W.attn_tensors(shape, 0)
    heads = 1
    for _ in range(args.warmup):
        oracle_sample(plan_o, q, k, v, do, shape.scale, heads)
    times = []
    flops = 0.0
    for _ in range(args.steps):
        dt, flops = oracle_sample(plan_o, q, k, v, do, shape.scale, heads)
        times.append(dt)
    tot = sum(times)
    val = flops * args.steps / tot / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"float64 NumPy oracle, fwd+bwd of {heads} of {shape.n_q_heads} query heads "
              f"(its kv head) over the whole packed row, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_DESC, "sample_heads": heads},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "trajectories_per_s": None,
    }
    print(json.dumps(line), flush=True)


PROFILE_CASES = ("attn", "classify", "index", "logprob", "gdn", "gdn_train")


def profile_case(name: str, reps: int) -> None:
    """Untimed calls of one component on the benchmarked workload (one warm
    call, then `reps`), for a profiler to capture: the command behind the
    ncu summaries.  The attention keeps the dS tiles of two kv-head groups at
    a time (results identical to all groups at once), so the case holds about
    1.5 GB on the device."""
    import torch

    from sft_trie_build_gb300 import stp

    dev = torch.device("cuda", 0)
    b = _batch(0)
    tokens, offsets, train = b.flat()
    plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=b.min_shared)
    info = stp.stp_plan_info(plan)
    R, T = info["n_rows"], info["row_len"]
    meta = stp.stp_plan_write(plan)
    shape = W.attn_shape(WORKLOAD, R, T)
    desc = stp.Desc(R, T, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, stp.STP_BF16, shape.scale,
                    stp.stp_count_tile_pairs(meta["subtree_end"]), ds_groups=2)
    buf = stp.Buffers(desc, dev)
    se = torch.from_numpy(np.ascontiguousarray(meta["subtree_end"])).to(dev)
    calls = []
    if name in ("attn", "classify"):
        q, k, v, do = (x.to(dev) for x in W.attn_tensors(shape, 17))
        o, dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        lse = torch.empty(R, shape.n_q_heads, T, dtype=torch.float32, device=dev)

        def attn():
            stp.stp_classify(desc, se, buf.tile_meta)
            if name == "attn":
                stp.stp_attn_fwd(desc, q, k, v, se, buf.tile_meta, o, lse, buf.fwd_ws)
                stp.stp_attn_bwd(desc, q, k, v, o, lse, do, se, buf.tile_meta, dq, dk, dv, buf.bwd_ws)
        calls.append(attn)
    elif name == "index":
        stp.stp_classify(desc, se, buf.tile_meta)
        q, k, w = (x.to(dev) for x in W.index_tensors(R, T, 8, 64, seed=23))
        idesc = stp.index_desc(R, T, 8, 64, 512, desc.max_tile_pairs)
        ws = torch.empty(stp.stp_index_workspace_size(idesc), dtype=torch.uint8, device=dev)
        idx = torch.empty(R, T, 512, dtype=torch.int32, device=dev)
        sc = torch.empty(R, T, 512, dtype=torch.float32, device=dev)
        calls.append(lambda: stp.stp_index_topk(idesc, q, k, w, se, buf.tile_meta, idx, sc, ws))
    elif name == "logprob":
        h, w = (x.to(dev) for x in W.logprob_tensors(R * T, 4096, 151936, seed=29))
        tok = torch.from_numpy(np.ascontiguousarray(meta["token_ids"])).to(dev)
        mask = torch.from_numpy(np.ascontiguousarray(meta["loss_mask"])).to(dev)
        ldesc = stp.logprob_desc(R, T, 4096, 151936)
        ws = torch.empty(stp.stp_logprob_workspace_size(ldesc), dtype=torch.uint8, device=dev)
        out = torch.empty(R * T, dtype=torch.float32, device=dev)
        calls.append(lambda: stp.stp_logprob_gather(ldesc, h, w, tok, mask, out, ws))
    else:   # gdn, gdn_train
        gi = np.asarray(meta["gather_index"])
        used = np.zeros(R, np.int64)
        np.maximum.at(used, gi // T, gi % T + 1)
        gdesc = stp.gdn_desc(R, T, 16)
        gplan = stp.stp_gdn_plan(gdesc, meta["subtree_end"], used.astype(np.int32))
        d_plan = torch.from_numpy(gplan).to(dev)
        x, cw, g, beta = (t.to(dev) for t in W.gdn_tensors(R * T, 16, 128, seed=31))
        o = torch.empty(R * T, 16, 128, dtype=torch.float32, device=dev)
        if name == "gdn":
            ws = torch.empty(stp.stp_gdn_workspace_size(gdesc, gplan), dtype=torch.uint8, device=dev)
            calls.append(lambda: stp.stp_gdn_fwd(gdesc, gplan, d_plan, x, cw, g, beta, o, ws))
        else:
            ws = torch.empty(stp.stp_gdn_train_workspace_size(gdesc, gplan), dtype=torch.uint8, device=dev)
            d_o = torch.randn(R * T, 16, 128, device=dev)
            dx = torch.empty(R * T, 3 * 16 * 128, device=dev)
            dw = torch.empty(3 * 16 * 128, 4, device=dev)
            dg = torch.empty(R * T, 16, device=dev)
            db = torch.empty(R * T, 16, device=dev)
            calls.append(lambda: stp.stp_gdn_fwd_train(gdesc, gplan, d_plan, x, cw, g, beta, o, ws))
            calls.append(lambda: stp.stp_gdn_bwd(gdesc, gplan, d_plan, x, cw, g, beta, d_o, dx, dw, dg, db, ws))
    for _ in range(1 + reps):
        for fn in calls:
            fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "calls": 1 + reps, "workload": WORKLOAD}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunks", type=int, default=8, help="kv-head groups of the host-buffer step")
    ap.add_argument("--profile", choices=PROFILE_CASES, default=None,
                    help="run one component untimed (1 + --reps calls) for a profiler; prints no bench line")
    ap.add_argument("--reps", type=int, default=1)
    args = ap.parse_args()
    if args.profile:
        profile_case(args.profile, args.reps)
        return

    peak, hbm, peak_kind = _peaks()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    from sft_trie_build_gb300 import stp

    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    b = _batch(rank)
    tokens, offsets, train = b.flat()
    plan0 = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len, min_shared=b.min_shared)
    info = stp.stp_plan_info(plan0)
    R, T = info["n_rows"], info["row_len"]
    shape = W.attn_shape(WORKLOAD, R, T)
    Hq, Hkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    q_h, k_h, v_h, do_h = W.attn_tensors(shape, 17 + rank)
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    q_h, k_h, v_h, do_h = (pin(x) for x in (q_h, k_h, v_h, do_h))
    q, k, v, do = (x.to(dev) for x in (q_h, k_h, v_h, do_h))
    meta0 = stp.stp_plan_write(plan0)
    se0 = meta0["subtree_end"]
    desc = stp.Desc(R, T, Hq, Hkv, D, stp.STP_BF16, shape.scale, stp.stp_count_tile_pairs(se0))
    buf = stp.Buffers(desc, dev)
    o = torch.empty_like(q)
    lse = torch.empty(R, Hq, T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # Two pinned sets of row metadata: the host packs batch i + 1 into one
    # while the upload of batch i from the other is in flight (the way a data
    # loader prepares the next batch during the current step).
    meta_h, meta_np = [], []
    for _ in range(2):
        mh = {n: torch.empty(R, T, dtype=torch.int32).pin_memory() for n in
              ("token_ids", "position_ids", "subtree_end")}
        mn = {n: t.numpy() for n, t in mh.items()}
        mn["loss_mask"] = torch.empty(R, T, dtype=torch.uint8).pin_memory().numpy()
        mn["gather_index"] = np.empty(int(offsets[-1]), np.int64)
        meta_h.append(mh)
        meta_np.append(mn)
    up_done = [torch.cuda.Event(), torch.cuda.Event()]
    meta_d = {n: torch.empty(R, T, dtype=torch.int32, device=dev) for n in meta_h[0]}
    se = meta_d["subtree_end"]
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    useful = float(info["useful_pairs"])
    fwd_flops = 4.0 * D * Hq * useful
    bwd_flops = 10.0 * D * Hq * useful
    step_flops = fwd_flops + bwd_flops
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    pack_ms = []

    def pack(x):
        """Host: plan the batch and write its rows into metadata set x (once
        the upload that last read set x has finished)."""
        up_done[x].synchronize()
        t0 = time.perf_counter()
        plan = stp.stp_pack(tokens, offsets, train, b.family, row_len=b.row_len,
                            min_shared=b.min_shared)
        stp.stp_plan_write(plan, meta_np[x])
        pack_ms.append(1e3 * (time.perf_counter() - t0))
        return plan

    def upload(x):
        for n in meta_d:
            meta_d[n].copy_(meta_h[x][n], non_blocking=True)
        up_done[x].record()

    def attention(marks=None):
        stp.stp_classify(desc, se, buf.tile_meta)
        if marks:
            marks[0].record()
        stp.stp_attn_fwd(desc, q, k, v, se, buf.tile_meta, o, lse, buf.fwd_ws)
        if marks:
            marks[1].record()
        stp.stp_attn_bwd(desc, q, k, v, o, lse, do, se, buf.tile_meta, dq, dk, dv, buf.bwd_ws)
        if marks:
            marks[2].record()

    # ---- device leg: inputs resident in HBM.  Every step packs its batch on
    # the host (into the free metadata set, while the GPU runs the previous
    # step), uploads the rows, classifies, and runs forward and backward.
    cur = 0
    pack(cur)
    for _ in range(args.warmup):
        upload(cur)
        attention()
        cur ^= 1
        pack(cur)
    torch.cuda.synchronize()
    for ws in (buf.tile_meta, buf.fwd_ws, buf.bwd_ws):
        assert stp.stp_device_status(ws) == stp.STP_OK
    sampler = ClockSampler(_gpu_id(torch, local))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)   # nvidia-smi's first sample
    t_start = time.time()
    steps = []
    pack_ms.clear()
    for i in range(args.steps):
        flush.fill_(1)  # L2 flushed on the GPU before every step, outside its events
        s0, f0, f1, b1, s1 = ev(), ev(), ev(), ev(), ev()
        s0.record()
        upload(cur)
        attention((f0, f1, b1))
        s1.record()
        steps.append((s0, f0, f1, b1, s1))
        cur ^= 1
        pack(cur)  # the next step's batch, while this one runs
    torch.cuda.synchronize()
    t_end = time.time()
    clocks = sampler.stop(t_start, t_end)
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(e) for a, _, _, _, e in steps]
    fwd_ms = [f0.elapsed_time(f1) for _, f0, f1, _, _ in steps]
    bwd_ms = [f1.elapsed_time(b1) for _, _, f1, b1, _ in steps]
    head_ms = [a.elapsed_time(f0) for a, f0, _, _, _ in steps]  # upload + classify
    host_pack_ms = statistics.mean(pack_ms)
    tot_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = tot_ms / args.steps
    value = world * step_flops * args.steps / (tot_ms / 1e3) / 1e12
    assert stp.stp_device_status(buf.bwd_ws) == stp.STP_OK

    # ---- end-to-end leg: host buffers in, gradients and O back to host
    o_h = torch.empty_like(q_h).pin_memory()
    dq_h, dk_h, dv_h = (torch.empty_like(x).pin_memory() for x in (q_h, k_h, v_h))
    h2d = sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h, do_h)) + \
        sum(x.numel() * x.element_size() for x in meta_h[0].values())
    d2h = sum(x.numel() * x.element_size() for x in (o_h, dq_h, dk_h, dv_h))

    # The host-buffer step of the library: uploads, kernels and downloads
    # pipelined over groups of kv heads on the library's own streams.  As in a
    # training loop, two steps are in flight: step i + 1 (its own caller
    # stream, scratch, tile metadata and pinned outputs) starts uploading while
    # step i still computes and downloads.  Every step uploads all of its
    # inputs and downloads all of its results; the timed region is the whole
    # run of K steps.
    n_chunks = args.chunks
    lse_h = torch.empty(R, Hq, T, dtype=torch.float32).pin_memory()
    d2h += lse_h.numel() * lse_h.element_size()
    lanes = []
    for k2 in range(2):
        outs = (o_h, lse_h, dq_h, dk_h, dv_h) if k2 == 0 else \
            tuple(torch.empty_like(x).pin_memory() for x in (o_h, lse_h, dq_h, dk_h, dv_h))
        lanes.append({
            "stream": torch.cuda.Stream(dev),
            "scratch": torch.empty(stp.stp_step_scratch_size(desc, n_chunks), dtype=torch.uint8, device=dev),
            "tile_meta": torch.empty_like(buf.tile_meta),
            "meta": {n: torch.empty_like(t) for n, t in meta_d.items()},
            "outs": outs,
        })

    def e2e_step(x, lane):
        st = lane["stream"]
        with torch.cuda.stream(st):
            for n, t in lane["meta"].items():
                t.copy_(meta_h[x][n], non_blocking=True)
            up_done[x].record(st)
            se_l = lane["meta"]["subtree_end"]
            stp.stp_classify(desc, se_l, lane["tile_meta"], stream=st)
            stp.stp_attn_step_host(desc, n_chunks, q_h, k_h, v_h, do_h, se_l, lane["tile_meta"],
                                   *lane["outs"], lane["scratch"], stream=st)

    for i in range(args.warmup):
        e2e_step(cur, lanes[i % 2])
        cur ^= 1
        pack(cur)
    torch.cuda.synchronize()
    e_start, e_end, e_join = ev(), ev(), ev()
    e_start.record(lanes[0]["stream"])
    lanes[1]["stream"].wait_event(e_start)
    for i in range(args.steps):
        e2e_step(cur, lanes[i % 2])
        cur ^= 1
        pack(cur)
    e_join.record(lanes[1]["stream"])
    lanes[0]["stream"].wait_event(e_join)
    e_end.record(lanes[0]["stream"])
    torch.cuda.synchronize()
    e_tot = max_over_ranks(e_start.elapsed_time(e_end), dev)
    for lane in lanes:
        assert stp.stp_device_status(lane["scratch"]) == stp.STP_OK
        assert torch.equal(lane["outs"][0], o.cpu()) and torch.equal(lane["outs"][1], lse.cpu()), \
            "host-buffer step differs"
    e2e_value = world * step_flops * args.steps / (e_tot / 1e3) / 1e12

    bwd_avg = statistics.mean(bwd_ms)
    achieved = bwd_flops / (bwd_avg / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "rows": R, "row_len": T, "sequences": b.n_seqs,
                   "useful_pairs_per_head": int(useful), "useful_tflop_per_step": step_flops / 1e12,
                   "packed_tokens": info["packed_tokens"], "input_tokens": info["input_tokens"],
                   "l2": "flushed (512 MiB write) before every timed step", "parallelism": f"replicas x{world}",
                   "host_pack": "every step packs its batch on the host (trie, placement, rows) while the GPU "
                                "runs the previous step; the first batch is packed before the timed region"},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "trajectories_per_s": world * b.n_seqs * args.steps / (tot_ms / 1e3),
        "breakdown_ms": {"host_pack_overlapped": host_pack_ms, "upload_classify": statistics.mean(head_ms),
                         "fwd": statistics.mean(fwd_ms),
                         "bwd": bwd_avg, "fwd_tflops": fwd_flops / (statistics.mean(fwd_ms) / 1e3) / 1e12,
                         "bwd_tflops": achieved},
        "roofline": {"bound": "tensor",
                     "kernel": "stp_attn_bwd call: bwd_delta_kernel + bwd_tc_kernel (dK, dV, dS tiles) + "
                               "dq_tc_kernel (dQ from the dS tiles)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} bf16 burst", "traffic": BWD_DRAM_BYTES,
                     "traffic_note": "dram read+write bytes of one backward call (Delta pass, 8 x dK/dV, "
                                     "8 x dQ) from one ncu capture; the dS round trip is ~7.8 GB of it"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e_tot / args.steps, "call": "stp_attn_step_host", "kv_head_groups": n_chunks,
                "steps_in_flight": 2, "l2": "not flushed: every step re-uploads 336 MB of inputs (> L2)"},
        # per step: four classification kernels, the forward, Delta, and dK/dV + dQ per kv-head group
        "gpu_launches": (6 + 2 * min(Hkv, 8)) * args.steps,
    }
    if rank == 0:
        line["classify"] = _classify_bandwidth(desc, se, buf.tile_meta)
        cfgs = {}
        for name in ("tiny", "curriculum", "deep", "bushy"):
            try:
                cfgs[name] = _attn_config(name, dev, peak, flush,
                                          oracle_heads=0 if args.no_cpu_baseline else 1)
            except Exception as exc:  # an auxiliary field: report, do not lose the bench line
                cfgs[name] = {"error": repr(exc)}
        line["configs"] = cfgs
        line["list_mode"] = _list_mode(dev, peak, flush)
        line["planning_cost"] = _planning_cost()
        line["what_if"] = _what_if()
        line["indexer"] = _indexer(R, T, se, buf.tile_meta, desc.max_tile_pairs, useful, dev)
        line["logprob"] = _logprob(meta0["token_ids"], meta0["loss_mask"], dev, peak)
        line["gdn"] = _gdn(meta0, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import pack as OP
        plan_o = OP.pack(b.seqs, b.trainable, b.row_len, b.min_shared, b.family)
        nh = 8
        dt, fl = oracle_sample(plan_o, q_h.float(), k_h.float(), v_h.float(), do_h.float(), shape.scale, nh)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle",
                                "sample": f"float64 NumPy oracle fwd+bwd of {nh} of {Hq} query heads "
                                          f"(their kv heads) over the whole packed row ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
