"""Runs stp_gdn_fwd on a packed plan and evaluates the oracle on the same inputs."""
import numpy as np
import torch

from oracle import gdn as OG
from sft_trie_build_gb300 import stp
from sft_trie_build_gb300 import workloads as W


def run_gdn(plan_o, H, seed=0, reps=1):
    R, T = plan_o.n_rows, plan_o.row_len
    desc = stp.gdn_desc(R, T, H)
    plan = stp.stp_gdn_plan(desc, plan_o.subtree_end, np.asarray(plan_o.used, np.int32))
    d_plan = torch.from_numpy(plan).cuda()
    x, cw, g, beta = W.gdn_tensors(R * T, H, 128, seed)
    ws = torch.empty(stp.stp_gdn_workspace_size(desc, plan), dtype=torch.uint8, device="cuda")
    o = torch.full((R * T, H, 128), float("nan"), device="cuda")
    args = (x.cuda(), cw.cuda(), g.cuda(), beta.cuda())
    outs = []
    for _ in range(reps):
        stp.stp_gdn_fwd(desc, plan, d_plan, *args, o, ws)
        torch.cuda.synchronize()
        outs.append(o.cpu().numpy().copy())
    return outs, stp.stp_device_status(ws), (x, cw, g, beta), desc.scale


def oracle_rows(plan_o, H, inputs, scale):
    x, cw, g, beta = inputs
    T = plan_o.row_len
    out = []
    for r in range(plan_o.n_rows):
        sl = slice(r * T, (r + 1) * T)
        out.append(OG.gdn_row(plan_o, r, x[sl].float().numpy(), cw.numpy(), g[sl].numpy(), beta[sl].numpy(),
                              H, 128, scale))
    return np.concatenate(out)


def oracle_sequence_heads(plan_o, seq_index, offsets, heads, inputs, scale):
    """Oracle outputs [len, len(heads), 128] of one sequence, unpacked, with the
    inputs read at its packed positions (gather_index)."""
    x, cw, g, beta = inputs
    idx = plan_o.gather_index[offsets[seq_index]: offsets[seq_index + 1]]
    xs = x[torch.from_numpy(idx)].float().numpy()
    L = len(idx)
    prev = np.arange(L) - 1
    y = OG.conv_path(xs, cw.numpy(), prev)
    H = g.shape[1]
    q, k, v = OG.split_heads(y, H, 128)
    outs = []
    for h in heads:
        outs.append(OG.delta_rule(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], g.numpy()[idx][:, h:h + 1],
                                  beta.numpy()[idx][:, h:h + 1], prev, scale)[:, 0])
    return np.stack(outs, 1), idx


def run_gdn_train(plan_o, H, seed=0):
    """Training forward + backward for L = sum dO . o, dO ~ N(0, 1) on real
    tokens and 0 on pads; returns (o, dx, dconv_w, dg, dbeta), the status,
    the inputs and dO."""
    R, T = plan_o.n_rows, plan_o.row_len
    desc = stp.gdn_desc(R, T, H)
    used = np.asarray(plan_o.used, np.int32)
    plan = stp.stp_gdn_plan(desc, plan_o.subtree_end, used)
    d_plan = torch.from_numpy(plan).cuda()
    x, cw, g, beta = W.gdn_tensors(R * T, H, 128, seed)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1000 + seed)
    dO = torch.randn(R * T, H, 128, generator=gen)
    real = torch.zeros(R * T, dtype=torch.bool)
    for r in range(R):
        real[r * T: r * T + int(used[r])] = True
    dO[~real] = 0.0
    ws = torch.empty(stp.stp_gdn_train_workspace_size(desc, plan), dtype=torch.uint8, device="cuda")
    dev = [t.cuda() for t in (x, cw, g, beta)]
    o = torch.empty(R * T, H, 128, device="cuda")
    dx = torch.empty(R * T, 3 * H * 128, device="cuda")
    dw = torch.empty(3 * H * 128, 4, device="cuda")
    dg = torch.empty(R * T, H, device="cuda")
    db = torch.empty(R * T, H, device="cuda")
    stp.stp_gdn_fwd_train(desc, plan, d_plan, *dev, o, ws)
    stp.stp_gdn_bwd(desc, plan, d_plan, *dev, dO.cuda(), dx, dw, dg, db, ws)
    torch.cuda.synchronize()
    outs = tuple(t.cpu().numpy() for t in (o, dx, dw, dg, db))
    return outs, stp.stp_device_status(ws), (x, cw, g, beta), dO.numpy(), desc.scale


def oracle_row_grads(plan_o, H, inputs, dO, scale):
    """(dx, dconv_w, dg, dbeta) of the oracle over every row of the plan."""
    x, cw, g, beta = inputs
    T = plan_o.row_len
    dxs, dgs, dbs, dw = [], [], [], 0.0
    for r in range(plan_o.n_rows):
        sl = slice(r * T, (r + 1) * T)
        gx, gw, gg, gb = OG.gdn_row_grads(plan_o, r, x[sl].float().numpy(), cw.numpy(), g[sl].numpy(),
                                          beta[sl].numpy(), dO[sl], H, 128, scale)
        dxs.append(gx)
        dgs.append(gg)
        dbs.append(gb)
        dw = dw + gw
    return np.concatenate(dxs), dw, np.concatenate(dgs), np.concatenate(dbs)


def oracle_head_grads(plan_o, r, inputs, dO, scale, H, heads):
    """Oracle gradients of row r for some heads only: heads never mix in the
    layer core (the convolution is per channel), so head h is the layer with
    H = 1 on its own q, k, v channels.  {h: (channels, dx, dconv_w, dg, dbeta)}."""
    x, cw, g, beta = inputs
    T = plan_o.row_len
    sl = slice(r * T, (r + 1) * T)
    out = {}
    for h in heads:
        ch = np.concatenate([np.arange(b * H * 128 + h * 128, b * H * 128 + (h + 1) * 128) for b in range(3)])
        gx, gw, gg, gb = OG.gdn_row_grads(plan_o, r, x[sl][:, ch].float().numpy(), cw.numpy()[ch],
                                          g[sl][:, [h]].numpy(), beta[sl][:, [h]].numpy(), dO[sl][:, [h]],
                                          1, 128, scale)
        out[h] = (ch, gx, gw, gg[:, 0], gb[:, 0])
    return out
