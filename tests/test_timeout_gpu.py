"""A device-side wait that runs out of time is reported, not hung or faulted.

The fused dispatch's grid-barrier waits are bounded; moe_set_barrier_wait_limit_ns
shortens the bound. With a 1 ns limit on a launch where blocks reach the first
barrier at different times (16384 tokens in 586 tiles over one block per SM, so
blocks route 3 or 4 tiles each), the early blocks give up, record the timeout
and return. Nothing waits on anything that cannot end: every wait stays
bounded, and no TMA copy is in flight in this kernel. The host then reads
MOE_ERR_TIMEOUT, and the next launch with the default limit is clean and
matches the oracle's route, layout and permute."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth

from _parity import assert_close, assert_equal, desc_of, np64, npi, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


def fused(d, b):
    moe.moe_dispatch_fused(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.cnt, b.off, b.slot,
                           b.row_src, b.cnt_re, b.rank_off, b.x_perm, b.ws)


def test_barrier_timeout_is_reported_and_the_next_launch_is_clean():
    inp = moe_synth.make_inputs(T=16384, H=256, E=64, k=4, F=64, R=8, seed=71)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    torch.cuda.synchronize()
    old = moe.moe_set_barrier_wait_limit_ns(1)
    try:
        fused(d, b)
        st = moe.moe_device_status(d, b.ws)
    finally:
        prev = moe.moe_set_barrier_wait_limit_ns(0)
    assert prev == 1
    assert old == 2_000_000_000
    assert st == moe.MOE_ERR_TIMEOUT, moe.lib().moe_last_error()
    # the status words were cleared by the read; the default limit is back
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    for t in (b.idx, b.slot, b.row_src, b.cnt, b.off, b.x_perm):
        t.fill_(0)
    fused(d, b)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    o = oracle_layer(inp)
    T, k = inp.T, inp.k
    N = T * k
    assert_equal("logits", b.logits.cpu().numpy().view(np.uint32),
                 np.asarray(o["z"], np.float32).view(np.uint32))
    for key in ("idx", "slot"):
        assert_equal(key, npi(getattr(b, key)), o[key])
    for key in ("cnt", "off", "cnt_re", "rank_off"):
        assert_equal(key, npi(getattr(b, key)), o[key])
    assert_equal("row_src", npi(b.row_src)[:N], o["row_src"])
    assert_equal("x_perm", np64(b.x_perm)[:N], o["x_perm"])
    assert_close("gates", np64(b.gates), o["gates"], tol=1e-5)
