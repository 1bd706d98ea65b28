"""The multi-process path of bench.py on CPU: two gloo ranks, rendezvous on
127.0.0.1, barrier and max-over-ranks timing (the slowest rank sets the time).

bench.py runs one independent replica per GPU (no collective on the data
path); the process group only aligns the timed region and reduces the time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(float(rank + 1), w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        assert dict(out) == {0: 2.0, 1: 2.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(key, raising=False)
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
