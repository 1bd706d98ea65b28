"""CPU oracle of the expert-parallel (EP) exchange around one MoE layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module; only
the tests do. It shares no code with the CUDA path or with the package's
exchange module: it uses ``moe_oracle`` for the layer's own arithmetic and
plain numpy for the exchange.

What the pages fix: the dispatcher is the standard MoE all-to-all ("MoE
expert-parallel overlap" skill card, section "what it is", dispatcher table),
run across 16 ranks in the production benchmark (EP16, skill card sections
"HybridEP production benchmark" and the correctness-first all-to-all
benchmark). Each rank owns E/R experts; the "1. MoE EP Overlap" note splits the
layer into dispatch -> mlp -> combine, with dispatch and combine being the
exchange. The pages give no data layout, so these readings are taken (each is
also listed in the design notes):
  R14 ranks and experts: rank d owns experts d*E_l .. (d+1)*E_l - 1, E_l = E/R;
      every rank routes its own tokens with the same router and sends each
      routed row to the owner of its expert.
  R15 send buffer: a rank's permuted buffer (dispatch layout R5) is rank-major
      and expert-contiguous; rows rank_off[d] .. rank_off[d+1]-1 go to rank d,
      preceded by the counts cnt_re[d][:] (one per local expert of d).
  R16 receive order: a rank receives the chunks of sources s = 0..R-1 in source
      order, each chunk ordered by local expert and, inside an expert, as the
      source sent it (ascending token). recv_cnt[s][l] = cnt_re of source s,
      row d. This is what an all-to-allv with per-source splits delivers.
  R17 re-sort: before the grouped GEMM the receiver reorders its rows
      expert-major: local expert l first, then, inside l, source s ascending,
      then the source's own order. The expert's offsets are off_local[l] =
      sum over l' < l and all s of recv_cnt[s][l']. The inverse re-sort puts
      expert-major rows (o, dx_perm) back in receive order for the return
      exchange, which is the dispatch exchange mirrored.
With these readings the rows of expert e on its owner are the rows of e in the
single-rank layout of all ranks' tokens concatenated in rank order, in the
same order: the EP layer equals the single-rank layer on those tokens, which
the pins check.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as O

__all__ = ["exchange_counts", "resort_offsets", "ep_resort", "ep_unsort", "ep_layer"]


def exchange_counts(cnt_re_all):
    """Count exchange. cnt_re_all[s] is source s's [R, E_l] table (rows it sends
    to rank d's local expert l). Returns recv_cnt_all[d] = [R, E_l] with
    recv_cnt_all[d][s][l] = cnt_re_all[s][d][l] (R16)."""
    R = len(cnt_re_all)
    return [np.stack([np.asarray(cnt_re_all[s])[d] for s in range(R)]) for d in range(R)]


def resort_offsets(recv_cnt):
    """Offsets of the two orders of one receiver's rows (R16, R17).

    recv_cnt [R, E_l]. Returns (src_off, dst_off, off_local):
      src_off[s][l]: first row of (s, l) in receive order (source-major);
      dst_off[s][l]: first row of (s, l) in expert-major order;
      off_local [E_l + 1]: first row of each local expert, expert-major."""
    c = np.asarray(recv_cnt, np.int64)
    R, E_l = c.shape
    src_off = np.zeros((R, E_l), np.int64)
    dst_off = np.zeros((R, E_l), np.int64)
    run = 0
    for s in range(R):          # receive order: source, then expert
        for l in range(E_l):
            src_off[s, l] = run
            run += c[s, l]
    off_local = np.zeros(E_l + 1, np.int64)
    run = 0
    for l in range(E_l):        # expert-major: expert, then source
        off_local[l] = run
        for s in range(R):
            dst_off[s, l] = run
            run += c[s, l]
    off_local[E_l] = run
    return src_off, dst_off, off_local


def ep_resort(recv, recv_cnt):
    """Receive order -> expert-major order (R17): out[dst_off[s,l] + i] =
    recv[src_off[s,l] + i] for i < recv_cnt[s,l]. Returns (out, off_local)."""
    recv = np.asarray(recv)
    src_off, dst_off, off_local = resort_offsets(recv_cnt)
    c = np.asarray(recv_cnt, np.int64)
    out = np.empty_like(recv)
    for s in range(c.shape[0]):
        for l in range(c.shape[1]):
            n = c[s, l]
            out[dst_off[s, l]:dst_off[s, l] + n] = recv[src_off[s, l]:src_off[s, l] + n]
    return out, off_local


def ep_unsort(buf, recv_cnt):
    """Expert-major order -> receive order (the inverse of ep_resort)."""
    buf = np.asarray(buf)
    src_off, dst_off, _ = resort_offsets(recv_cnt)
    c = np.asarray(recv_cnt, np.int64)
    out = np.empty_like(buf)
    for s in range(c.shape[0]):
        for l in range(c.shape[1]):
            n = c[s, l]
            out[src_off[s, l]:src_off[s, l] + n] = buf[dst_off[s, l]:dst_off[s, l] + n]
    return out


def _exchange(send_all, rank_off_all):
    """All-to-allv: receiver d gets, for s = 0..R-1, rows rank_off_s[d]..rank_off_s[d+1]-1
    of source s's buffer, concatenated in source order (R16)."""
    R = len(send_all)
    return [np.concatenate([np.asarray(send_all[s])[rank_off_all[s][d]:rank_off_all[s][d + 1]]
                            for s in range(R)]) for d in range(R)]


def _return(back_all, rank_off_all):
    """The mirrored exchange: receiver d's buffer in receive order is cut by
    source and each piece goes back to rows rank_off_s[d].. of source s."""
    R = len(back_all)
    out = []
    for s in range(R):
        pieces = []
        for d in range(R):
            start = sum(int(rank_off_all[s2][d + 1] - rank_off_all[s2][d]) for s2 in range(s))
            n = int(rank_off_all[s][d + 1] - rank_off_all[s][d])
            pieces.append(np.asarray(back_all[d])[start:start + n])
        out.append(np.concatenate(pieces))
    return out


def ep_layer(inps, R: int, rnd=O.bf16_rne):
    """One MoE layer, forward and backward, over R ranks with the EP exchange.

    inps[r] holds rank r's tokens (x, dy) and the shared weights (w_r, w1, w2,
    bias); every input has E experts and R ranks. Each rank routes and lays
    out its own tokens (moe_oracle), the send buffers are exchanged (R15,
    R16), each owner re-sorts expert-major (R17) and runs its local experts
    forward, dgrad and wgrad; the outputs o and dx_perm go back by the inverse
    re-sort and the mirrored exchange, and each source combines and runs the
    dispatch and router backward on its own tokens. Returns per-rank dicts with
    the source-side results (y, dx, dw_r, idx, gates, layout) and the owner-side
    ones (recv_cnt, off_local, x_recv expert-major, dw1/dw2 of the local
    experts)."""
    assert len(inps) == R
    E = inps[0].E
    E_l = E // R
    k = inps[0].k
    w1, w2 = O._np(inps[0].w1), O._np(inps[0].w2)
    src = []
    for inp in inps:
        x, w_r = O._np(inp.x), O._np(inp.w_r)
        bias = None if inp.bias is None else O._np(inp.bias)
        z = O.router_logits_fp32(x, w_r, bias)
        idx, gates = (O.route_forced if inp.mode == 1 else O.route_topk)(z, k)
        lay = O.dispatch_layout(idx, E, R)
        src.append(dict(x=x, z=z, idx=idx, gates=gates, x_perm=O.permute(x, lay["row_src"], k),
                        **lay))
    rank_off_all = [s["rank_off"] for s in src]
    recv_cnt_all = exchange_counts([s["cnt_re"] for s in src])
    # forward: dispatch exchange, re-sort, local experts, inverse re-sort, return
    x_recv = _exchange([s["x_perm"] for s in src], rank_off_all)
    own = []
    for d in range(R):
        xs, off_l = ep_resort(x_recv[d], recv_cnt_all[d])
        ex = slice(d * E_l, (d + 1) * E_l)
        a, h, o = O.expert_ffn_fwd(xs, off_l, w1[ex], w2[ex], rnd)
        own.append(dict(recv_cnt=recv_cnt_all[d], off_local=off_l, x_sorted=xs, a=a, h=h, o=o))
    o_back = _return([ep_unsort(w["o"], w["recv_cnt"]) for w in own], rank_off_all)
    for r, s in enumerate(src):
        s["o"] = o_back[r]
        s["y"] = O.combine(s["o"], s["slot"], s["gates"], rnd)
    # backward: combine backward at the source, the same exchange for d_o
    for r, s in enumerate(src):
        s["d_o"], s["dgates"] = O.combine_bwd(O._np(inps[r].dy), s["o"], s["slot"], s["gates"],
                                              rnd)
    do_recv = _exchange([s["d_o"] for s in src], rank_off_all)
    for d, w in enumerate(own):
        ex = slice(d * E_l, (d + 1) * E_l)
        w["d_o"], _ = ep_resort(do_recv[d], w["recv_cnt"])
        w["da"], w["dx_perm"] = O.expert_ffn_bwd_dgrad(w["d_o"], w["a"], w["off_local"], w1[ex],
                                                       w2[ex], rnd)
        w["dw1"], w["dw2"] = O.expert_ffn_bwd_wgrad(w["x_sorted"], w["h"], w["d_o"], w["da"],
                                                    w["off_local"], E_l, rnd)
    dxp_back = _return([ep_unsort(w["dx_perm"], w["recv_cnt"]) for w in own], rank_off_all)
    for r, s in enumerate(src):
        s["dx_perm"] = dxp_back[r]
        dx_e = O.permute_bwd(s["dx_perm"], s["slot"])
        s["dz"], s["dx"], s["dw_r"] = O.route_bwd(s["dgates"], s["z"], s["idx"], s["x"],
                                                  O._np(inps[r].w_r), dx_e, rnd)
    return dict(src=src, own=own, x_recv=x_recv)
