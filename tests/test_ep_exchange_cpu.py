"""The expert-parallel exchange (combine_router_softmax_top_gb300.ep) among
world-size-2 gloo ranks on the CPU, against the EP oracle.

Each rank lays out its own tokens (the layout comes from the oracle here: the
ranks have no GPU), then the package's exchange code moves the counts and the
send buffer with torch.distributed all-to-alls. What a rank receives must be,
bit for bit, the oracle's receive-order rows and counts; after the owner's
expert outputs come back through the mirrored exchange, each source must hold
the oracle's o in its own send-buffer order."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(R, T_list, E, k, bias):
    import moe_synth
    H, F = 32, 16
    base = moe_synth.make_inputs(T=sum(T_list), H=H, E=E, k=k, F=F, R=R, bias=bias, seed=77)
    inps, t0 = [], 0
    for T in T_list:
        inp = moe_synth.make_inputs(T=T, H=H, E=E, k=k, F=F, R=R, bias=bias, seed=77)
        inp.x = base.x[t0:t0 + T].contiguous()
        inp.dy = base.dy[t0:t0 + T].contiguous()
        inps.append(inp)
        t0 += T
    return inps


def _rank(rank, world, port, T_list, E, k, bias, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from combine_router_softmax_top_gb300 import ep
    from oracle import ep_oracle as EP
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inps = _inputs(world, T_list, E, k, bias)
        want = EP.ep_layer(inps, world)  # every rank knows the whole expected exchange
        me = want["src"][rank]
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)  # noqa: E731
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.int32)  # noqa: E731
        send = bf(me["x_perm"])
        recv, recv_cnt, s_out, s_in = ep.dispatch(send, i32(me["cnt_re"]), i32(me["rank_off"]))
        own = want["own"][rank]
        res = {
            "recv_cnt": bool(np.array_equal(recv_cnt.numpy(), own["recv_cnt"])),
            "recv": bool(np.array_equal(recv.to(torch.float64).numpy(), want["x_recv"][rank])),
            "splits": s_out == np.diff(me["rank_off"]).tolist()
                      and s_in == own["recv_cnt"].sum(1).tolist(),
        }
        # the owner's expert outputs, back in receive order, return to their sources
        back = bf(EP.ep_unsort(own["o"], own["recv_cnt"]))
        o_src = ep.combine_return(back, s_out, s_in)
        res["o_back"] = bool(np.array_equal(o_src.to(torch.float64).numpy(), me["o"]))
        res["rows"] = int(recv.shape[0])
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T_list,E,k,bias", [([40, 25], 8, 2, None),
                                             ([50, 3], 16, 4, "zipf_logrank")])
def test_two_rank_exchange_matches_the_oracle(T_list, E, k, bias):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, T_list, E, k, bias, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        res = dict(out)
    for r in range(world):
        assert res[r]["recv_cnt"] and res[r]["recv"] and res[r]["splits"], (r, res[r])
        assert res[r]["o_back"], (r, res[r])
    assert sum(res[r]["rows"] for r in range(world)) == sum(T_list) * k
