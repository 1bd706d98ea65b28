"""The fused dispatch (moe_dispatch_fused: route, dispatch layout and permute in
one cooperative launch) gives the same bits as moe_route, moe_dispatch_layout
and moe_permute called one after the other, and matches the oracle."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth
from oracle import moe_oracle as O

from _parity import assert_equal, desc_of, np64, npi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


OUTS = ("logits", "idx", "gates", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off", "x_perm")


def three_calls(d, b):
    moe.moe_route(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.ws)
    moe.moe_dispatch_layout(d, b.idx, b.cnt, b.off, b.slot, b.row_src, b.cnt_re, b.rank_off,
                            b.ws)
    moe.moe_permute(d, b.x, b.row_src, b.x_perm)


def fused(d, b):
    moe.moe_dispatch_fused(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.cnt, b.off, b.slot,
                           b.row_src, b.cnt_re, b.rank_off, b.x_perm, b.ws)


CASES = {
    # one tile per block, ragged last tile
    "ragged": dict(T=301, H=192, E=16, k=3, F=64, seed=61),
    # the balanced routing of the benchmark, at a small hidden size
    "forced_4096": dict(T=4096, H=128, E=128, k=8, F=64, seed=62,
                        mode=moe_synth.ROUTE_FORCED_BALANCED),
    # several tiles per block (more tiles than resident blocks), R > 1 rank tables
    "many_tiles": dict(T=20000, H=64, E=32, k=2, F=64, R=4, seed=63),
    # skewed bias: empty experts and one expert taking most rows
    "skewed": dict(T=700, H=256, E=64, k=4, F=64, seed=64, bias="zipf_logrank"),
    # one token; k = E
    "one_token": dict(T=1, H=64, E=8, k=8, F=64, seed=65),
    # more experts than one block routes: the three separate launches
    "e256_fallback": dict(T=200, H=128, E=256, k=8, F=64, seed=66),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_matches_three_calls_and_oracle(case):
    inp = moe_synth.make_inputs(**CASES[case])
    d = desc_of(inp)
    ref, got = moe.LayerBuffers(d), moe.LayerBuffers(d)
    ref.load_inputs(inp)
    got.load_inputs(inp)
    for t in (got.idx, got.slot, got.row_src, got.x_perm, got.cnt, got.off):
        t.fill_(-7)  # every output must be written
    three_calls(d, ref)
    l0 = moe.moe_kernel_launches()
    fused(d, got)
    launches = moe.moe_kernel_launches() - l0
    torch.cuda.synchronize()
    assert moe.moe_device_status(d, got.ws) == moe.MOE_OK
    # one launch, or the separate router, layout and permute launches
    assert launches == 1 if inp.E <= 128 else launches > 1
    N = inp.T * inp.k
    for n in OUTS:
        a, b = getattr(ref, n), getattr(got, n)
        if n in ("row_src", "x_perm"):
            a, b = a[:N], b[:N]
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), n
    # against the oracle's layout and permute of the same routing
    o_lay = O.dispatch_layout(npi(got.idx)[: inp.T], inp.E, inp.R)
    for key in ("cnt", "off", "slot", "row_src", "cnt_re", "rank_off"):
        assert_equal(key, npi(getattr(got, key))[: len(o_lay[key])], o_lay[key])
    x_perm = O.permute(O._np(inp.x), o_lay["row_src"], inp.k)
    assert np.array_equal(np64(got.x_perm)[:N], x_perm)


def test_fused_dispatch_repeats_with_the_same_bits():
    """The grid barrier's counter is reset by every launch."""
    inp = moe_synth.make_inputs(T=1000, H=128, E=32, k=4, F=64, seed=67)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    fused(d, b)
    first = [getattr(b, n).clone() for n in OUTS]
    for _ in range(3):
        fused(d, b)
    torch.cuda.synchronize()
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    for n, a in zip(OUTS, first):
        assert torch.equal(a.view(torch.uint8), getattr(b, n).view(torch.uint8)), n
