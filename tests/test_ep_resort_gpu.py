"""The expert-parallel receive re-sort kernel (moe_ep_resort) against the EP
oracle, and a whole expert-parallel layer of two ranks emulated on one GPU.

The re-sort is a row copy, so it must match the oracle bit for bit, in both
directions, with empty (source, expert) pairs and sources that send nothing.
The emulated layer runs every step through the library's C ABI: each rank's
fused dispatch writes its send buffer and rank tables, the owner re-sorts the
rows it receives and runs its experts, the inverse re-sort and the return
bring o back, and the source combines; the backward mirrors it. Only the
all-to-all itself is emulated, by copying slices between the two ranks'
buffers (the package's exchange module runs it over torch.distributed, which
the gloo test covers on the CPU)."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth
from oracle import ep_oracle as EP

from _parity import assert_close, assert_equal, np64, npi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


@pytest.mark.parametrize("R,El,H,seed", [(2, 3, 256, 0), (8, 8, 128, 1), (4, 64, 64, 2),
                                         (1, 16, 2048, 3), (16, 1, 192, 4)])
def test_resort_matches_the_oracle_both_ways(R, El, H, seed):
    g = np.random.default_rng(seed)
    cnt = g.integers(0, 40, size=(R, El)).astype(np.int32)
    cnt[g.random((R, El)) < 0.2] = 0
    cnt[g.integers(0, R), :] = 0  # a source that sends nothing
    n = int(cnt.sum())
    d = moe.LayerDesc.of(T=1, H=H, E=R * El, k=1, F=64, R=R)
    x = torch.randn(max(n, 1), H, dtype=torch.float32).to(torch.bfloat16)
    want, want_off = EP.ep_resort(x[:n].float().numpy(), cnt)
    dx, dcnt = x.cuda(), torch.from_numpy(cnt).cuda()
    out = torch.full_like(dx, 7.0)
    off = torch.full((El + 1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_ep_resort(d, dcnt, dx, out, off)
    torch.cuda.synchronize()
    assert_equal("off_local", npi(off), want_off)
    assert_equal("expert-major", out[:n].float().cpu().numpy(), want)
    back = torch.full_like(dx, 7.0)
    moe.moe_ep_resort(d, dcnt, out, back, None, inverse=True)
    torch.cuda.synchronize()
    assert_equal("receive order", back[:n].float().cpu().numpy(), x[:n].float().numpy())


def test_resort_moves_nothing_past_the_buffer():
    """Counts that add up to more rows than the buffers hold: rows placed at or
    beyond n_rows are not moved, and no output row past n_rows is written."""
    R, El, H = 2, 2, 64
    cnt = np.array([[3, 2], [4, 1]], np.int32)  # 10 rows of counts
    n = 6
    d = moe.LayerDesc.of(T=1, H=H, E=R * El, k=1, F=64, R=R)
    x = torch.randn(n + 4, H).to(torch.bfloat16).cuda()
    x[n:] = 99.0
    out = torch.full_like(x, 5.0)
    moe.moe_ep_resort(d, torch.from_numpy(cnt).cuda(), x[:n], out[:n])
    torch.cuda.synchronize()
    full, _ = EP.ep_resort(np.arange(10)[:, None], cnt)  # source row of each output row
    src = full[:, 0]
    got = out.float().cpu().numpy()
    for o in range(n):
        if src[o] < n:
            assert np.array_equal(got[o], x[src[o]].float().cpu().numpy()), o
        else:
            assert np.all(got[o] == 5.0), o
    assert np.all(got[n:] == 5.0)


def _dev(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()


def test_two_ranks_emulated_on_one_gpu_match_the_ep_oracle():
    R, E, k, H, F = 2, 8, 2, 256, 128
    T_list = [96, 70]
    base = moe_synth.make_inputs(T=sum(T_list), H=H, E=E, k=k, F=F, R=R, seed=81)
    inps, t0 = [], 0
    for T in T_list:
        inp = moe_synth.make_inputs(T=T, H=H, E=E, k=k, F=F, R=R, seed=81)
        inp.x, inp.dy = base.x[t0:t0 + T].contiguous(), base.dy[t0:t0 + T].contiguous()
        inps.append(inp)
        t0 += T
    want = EP.ep_layer(inps, R)
    El = E // R
    # sources: route, lay out and permute their own tokens (the fused dispatch)
    src = []
    for inp in inps:
        d = moe.LayerDesc.of(**inp.shape_dict())
        b = moe.LayerBuffers(d)
        b.load_inputs(inp)
        moe.moe_dispatch_fused(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.cnt, b.off,
                               b.slot, b.row_src, b.cnt_re, b.rank_off, b.x_perm, b.ws)
        src.append((d, b))
    torch.cuda.synchronize()
    ro = [npi(b.rank_off) for _, b in src]
    cre = [b.cnt_re.clone() for _, b in src]

    def exchange(bufs):  # the all-to-allv, emulated: receiver d takes chunk d of each source
        return [torch.cat([bufs[s][ro[s][d]:ro[s][d + 1]] for s in range(R)]) for d in range(R)]

    def give_back(bufs):  # the mirrored exchange
        out = []
        for s in range(R):
            parts = []
            for d in range(R):
                start = sum(int(ro[s2][d + 1] - ro[s2][d]) for s2 in range(s))
                parts.append(bufs[d][start:start + int(ro[s][d + 1] - ro[s][d])])
            out.append(torch.cat(parts))
        return out

    recv_cnt = [torch.stack([cre[s][d] for s in range(R)]).contiguous() for d in range(R)]
    de = moe.LayerDesc.of(T=1, H=H, E=E, k=1, F=F, R=R)  # the re-sort's shape: all E, R ranks
    x_recv = exchange([b.x_perm[:int(ro[i][-1])] for i, (_, b) in enumerate(src)])
    owners = []
    for d in range(R):
        n = x_recv[d].shape[0]
        dd = moe.LayerDesc.of(T=max(n, 1), H=H, E=El, k=1, F=F, R=1)
        ob = moe.LayerBuffers(dd)
        ob.w1 = src[0][1].w1[d * El:(d + 1) * El]
        ob.w2 = src[0][1].w2[d * El:(d + 1) * El]
        off_l = torch.empty(El + 1, dtype=torch.int32, device="cuda")
        moe.moe_ep_resort(de, recv_cnt[d], x_recv[d], ob.x_perm, off_l)
        moe.moe_expert_ffn_fwd(dd, ob.x_perm, off_l, ob.w1, ob.w2, ob.a, ob.h, ob.o, ob.ws)
        back = torch.empty_like(ob.o)
        moe.moe_ep_resort(de, recv_cnt[d], ob.o, back, None, inverse=True)
        owners.append(dict(d=dd, b=ob, off=off_l, n=n, o_recv=back[:n]))
    o_src = give_back([w["o_recv"] for w in owners])
    for i, (d, b) in enumerate(src):
        b.o[:o_src[i].shape[0]].copy_(o_src[i])
        moe.moe_combine(d, b.o, b.slot, b.gates, b.y)
        moe.moe_combine_bwd(d, b.dy, b.o, b.slot, b.gates, b.d_o, b.dgates)
    do_recv = exchange([b.d_o[:int(ro[i][-1])] for i, (_, b) in enumerate(src)])
    for d, w in enumerate(owners):
        dd, ob = w["d"], w["b"]
        moe.moe_ep_resort(de, recv_cnt[d], do_recv[d], ob.d_o, None)
        moe.moe_expert_ffn_bwd_dgrad(dd, ob.d_o, ob.a, w["off"], ob.w1, ob.w2, ob.da, ob.dx_perm,
                                     ob.ws)
        moe.moe_expert_ffn_bwd_wgrad(dd, ob.x_perm, ob.h, ob.d_o, ob.da, w["off"], ob.dw1, ob.dw2,
                                     ob.ws)
        back = torch.empty_like(ob.dx_perm)
        moe.moe_ep_resort(de, recv_cnt[d], ob.dx_perm, back, None, inverse=True)
        w["dxp_recv"] = back[:w["n"]]
    dxp_src = give_back([w["dxp_recv"] for w in owners])
    for i, (d, b) in enumerate(src):
        b.dx_perm[:dxp_src[i].shape[0]].copy_(dxp_src[i])
        moe.moe_permute_bwd(d, b.dx_perm, b.slot, b.dx32)
        moe.moe_route_bwd(d, b.dgates, b.gates, b.idx, b.x, b.w_r, b.row_src, b.off, b.dx32, b.dx,
                          b.dw_r, b.ws)
    torch.cuda.synchronize()
    for i, (d, b) in enumerate(src):
        assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
        s = want["src"][i]
        assert_equal("idx", npi(b.idx), s["idx"])
        assert_equal("cnt_re", npi(b.cnt_re), s["cnt_re"])
        assert_equal("rank_off", npi(b.rank_off), s["rank_off"])
        assert_close("y", np64(b.y), s["y"])
        assert_close("dx", np64(b.dx), s["dx"])
        assert_close("dw_r", np64(b.dw_r), s["dw_r"])
    for d, w in enumerate(owners):
        o = want["own"][d]
        assert moe.moe_device_status(w["d"], w["b"].ws) == moe.MOE_OK
        assert_equal("recv_cnt", npi(recv_cnt[d]), o["recv_cnt"])
        assert_equal("off_local", npi(w["off"]), o["off_local"])
        assert_equal("x_sorted", np64(w["b"].x_perm)[:w["n"]], o["x_sorted"])
        assert_close("dw1", np64(w["b"].dw1), o["dw1"])
        assert_close("dw2", np64(w["b"].dw2), o["dw2"])
