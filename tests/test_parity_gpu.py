"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles and ragged tails, plus the degenerate cases of the layer."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth
from oracle import moe_oracle as O

from _parity import (assert_close, assert_equal, check_stages, compare_layer, desc_of, np64,
                     npi, oracle_layer, run_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


CASES = {
    # the tiny workload exactly as benchmarked
    "tiny": lambda: moe_synth.workload("tiny"),
    # ragged everything: T not a multiple of any tile, H and F not multiples of 128
    "ragged": lambda: moe_synth.make_inputs(T=300, H=192, E=6, k=3, F=192, seed=11),
    # several M tiles per expert and partial N tiles, R > 1 rank tables
    "multi_tile": lambda: moe_synth.make_inputs(T=1000, H=320, E=16, k=4, F=448, R=4, seed=12),
    # forced balancing, more experts than routed rows: most experts empty
    "empty_experts": lambda: moe_synth.make_inputs(T=5, H=128, E=16, k=2, F=128,
                                                   mode=moe_synth.ROUTE_FORCED_BALANCED, seed=13),
    # skewed bias with empty experts, k = E/2
    "skewed_small": lambda: moe_synth.make_inputs(T=512, H=256, E=32, k=16, F=256, seed=14,
                                                  bias="zipf_logrank"),
    # a single expert: the layer is a dense SwiGLU FFN
    "dense": lambda: moe_synth.make_inputs(T=130, H=128, E=1, k=1, F=128, seed=15),
    # every token to every expert
    "k_equals_E": lambda: moe_synth.make_inputs(T=70, H=128, E=4, k=4, F=128, seed=16),
    # one token
    "one_token": lambda: moe_synth.make_inputs(T=1, H=64, E=8, k=2, F=64, seed=17),
    # wide layer, deep K: several K stages and wide rows
    "wide": lambda: moe_synth.make_inputs(T=256, H=1024, E=8, k=2, F=512, seed=18),
    # the maximum expert count: two 128-expert router blocks, the separate top-k
    # kernel, 256-entry layout tables and tile prefixes
    "max_experts": lambda: moe_synth.make_inputs(T=200, H=128, E=256, k=8, F=64, seed=26),
    # k above 16: the 32-slot variants of the combine and router backward
    "large_k": lambda: moe_synth.make_inputs(T=150, H=192, E=32, k=20, F=64, seed=27),
    # the largest hidden size the header allows: 256 K stages in FC1 and the
    # router, 256 column slices in the dispatch backward, 32 KB rows
    "max_hidden": lambda: moe_synth.make_inputs(T=48, H=16384, E=4, k=2, F=128, seed=28),
    # the largest expert inner size: 128 FC1 column blocks, 256 K stages in FC2
    "max_inner": lambda: moe_synth.make_inputs(T=48, H=128, E=4, k=2, F=16384, seed=29),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_layer_parity(case):
    inp = CASES[case]()
    g = run_layer(inp)
    o = oracle_layer(inp)
    ew = {}
    errs = compare_layer(g, o, elementwise=ew)
    stages = check_stages(g, inp)
    print(case, {k: f"{v:.2e}" for k, v in errs.items()})
    print(case, "element-wise", {k: f"{v:.2e}" for k, v in ew.items()})
    print(case, "stages", {k: {m: f"{x:.2e}" for m, x in v.items()} for k, v in stages.items()})


def test_zero_tokens():
    inp = moe_synth.make_inputs(T=0, H=128, E=8, k=2, F=128, seed=19)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp) if inp.T else None
    b.w1.fill_(1.0)
    b.dw1.fill_(3.0)
    b.dw2.fill_(3.0)
    b.dw_r.fill_(3.0)
    moe.moe_layer_forward(d, b)
    moe.moe_layer_backward(d, b)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert npi(b.cnt).sum() == 0 and npi(b.off).sum() == 0
    assert float(b.dw1.abs().max()) == 0 and float(b.dw2.abs().max()) == 0
    assert float(b.dw_r.abs().max()) == 0


def test_entry_points_one_by_one():
    """Each entry point fed with the oracle's own inputs for that step."""
    inp = moe_synth.make_inputs(T=400, H=256, E=8, k=2, F=256, R=2, seed=21)
    o = oracle_layer(inp)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    dev = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(dt).cuda()  # noqa: E731
    N = inp.T * inp.k
    # route
    moe.moe_route(d, b.x, b.w_r, None, b.logits, b.idx, b.gates, b.ws)
    assert_equal("idx", npi(b.idx), o["idx"])
    assert_close("gates", np64(b.gates), o["gates"], tol=1e-5)
    # layout from the oracle's idx
    idx = dev(o["idx"], torch.int32)
    moe.moe_dispatch_layout(d, idx, b.cnt, b.off, b.slot, b.row_src, b.cnt_re, b.rank_off, b.ws)
    for key in ("cnt", "off", "slot", "row_src", "cnt_re", "rank_off"):
        assert_equal(key, npi(getattr(b, key))[: len(o[key])], o[key])
    # permute from the oracle's row_src
    row_src = dev(o["row_src"], torch.int32)
    moe.moe_permute(d, b.x, row_src, b.x_perm)
    assert_equal("x_perm", np64(b.x_perm)[:N], o["x_perm"])  # a copy: exact
    # experts from the oracle's x_perm
    off = dev(o["off"], torch.int32)
    x_perm = dev(o["x_perm"], torch.bfloat16)
    moe.moe_expert_ffn_fwd(d, x_perm, off, b.w1, b.w2, b.a, b.h, b.o, b.ws)
    for key in ("a", "h", "o"):
        assert_close(key, np64(getattr(b, key))[:N], o[key])
    # combine from the oracle's o, slot, gates
    slot = dev(o["slot"], torch.int32)
    gates = dev(o["gates"], torch.float32)
    o_dev = dev(o["o"], torch.bfloat16)
    moe.moe_combine(d, o_dev, slot, gates, b.y)
    assert_close("y", np64(b.y), o["y"], tol=1e-2)
    # combine backward
    moe.moe_combine_bwd(d, b.dy, o_dev, slot, gates, b.d_o, b.dgates)
    assert_close("d_o", np64(b.d_o)[:N], o["d_o"], tol=1e-2)
    assert_close("dgates", np64(b.dgates), o["dgates"], tol=1e-4)
    # dgrad from the oracle's d_o and a
    d_o = dev(o["d_o"], torch.bfloat16)
    a = dev(o["a"], torch.bfloat16)
    moe.moe_expert_ffn_bwd_dgrad(d, d_o, a, off, b.w1, b.w2, b.da, b.dx_perm, b.ws)
    assert_close("da", np64(b.da)[:N], o["da"])
    assert_close("dx_perm", np64(b.dx_perm)[:N], o["dx_perm"])
    # wgrad from the oracle's saved tensors
    h = dev(o["h"], torch.bfloat16)
    da = dev(o["da"], torch.bfloat16)
    moe.moe_expert_ffn_bwd_wgrad(d, x_perm, h, d_o, da, off, b.dw1, b.dw2, b.ws)
    assert_close("dw1", np64(b.dw1), o["dw1"])
    assert_close("dw2", np64(b.dw2), o["dw2"])
    # permute backward + router backward
    dx_perm = dev(o["dx_perm"], torch.bfloat16)
    moe.moe_permute_bwd(d, dx_perm, slot, b.dx32)
    assert_close("dx32", np64(b.dx32), o["dx_experts"], tol=1e-5)
    dgates = dev(o["dgates"], torch.float32)
    dx32 = dev(o["dx_experts"], torch.float32)
    moe.moe_route_bwd(d, dgates, gates, idx, b.x, b.w_r, row_src, off, dx32, b.dx, b.dw_r, b.ws)
    assert_close("dx", np64(b.dx), o["dx"], tol=1e-2)
    assert_close("dw_r", np64(b.dw_r), o["dw_r"], tol=1e-4)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK


def test_deterministic_run_to_run():
    inp = moe_synth.make_inputs(T=600, H=256, E=16, k=4, F=256, seed=23)
    g1 = run_layer(inp)
    g2 = run_layer(inp)
    for key in g1:
        assert np.array_equal(g1[key], g2[key]), key


def test_out_of_range_index_is_reported_not_faulted():
    inp = moe_synth.make_inputs(T=64, H=128, E=8, k=2, F=128, seed=24)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    bad = torch.zeros(64, 2, dtype=torch.int32, device="cuda")
    bad[:, 1] = 1
    bad[5, 0] = 99  # expert 99 does not exist
    moe.moe_dispatch_layout(d, bad, b.cnt, b.off, b.slot, b.row_src, b.cnt_re, b.rank_off, b.ws)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_ERR_INVALID_ARG
    assert int(b.slot[5, 0]) == -1
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK  # status words were cleared


def test_host_step_matches_device_path():
    inp = moe_synth.make_inputs(T=256, H=256, E=8, k=2, F=256, seed=25)
    g = run_layer(inp)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    hx = inp.x.clone().pin_memory()
    hdy = inp.dy.clone().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    b.x.zero_()
    b.dy.zero_()
    moe.moe_layer_step_host(d, b, hx, hdy, hy, hdx)
    assert np.array_equal(np64(hy), g["y"])
    assert np.array_equal(np64(hdx), g["dx"])


def test_pipelined_host_steps_match_single_steps():
    """moe_layer_steps_host over five different inputs (two buffer sets that
    share every buffer but x, dy, y and dx): each step's y and dx are the bits
    of the device path on that input, and the last step's weight gradients
    are that step's."""
    inps = [moe_synth.make_inputs(T=256, H=256, E=8, k=2, F=256, seed=25, microbatch=m)
            for m in range(5)]
    want = [run_layer(inp) for inp in inps]
    d = desc_of(inps[0])
    b0 = moe.LayerBuffers(d)
    b0.load_inputs(inps[0])
    b1 = moe.LayerBuffers(d, weights=b0)
    for name in ("logits", "idx", "gates", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off",
                 "x_perm", "a", "h", "o", "d_o", "dgates", "da", "dx_perm", "dx32", "dw_r", "dw1",
                 "dw2", "ws"):
        setattr(b1, name, getattr(b0, name))  # shared intermediates and gradients
    hx = [inp.x.clone().pin_memory() for inp in inps]
    hdy = [inp.dy.clone().pin_memory() for inp in inps]
    hy = [torch.empty_like(t).pin_memory() for t in hx]
    hdx = [torch.empty_like(t).pin_memory() for t in hx]
    moe.moe_layer_steps_host(d, b0, b1, hx, hdy, hy, hdx)
    for i in range(5):
        assert np.array_equal(np64(hy[i]), want[i]["y"]), i
        assert np.array_equal(np64(hdx[i]), want[i]["dx"]), i
    assert np.array_equal(np64(b0.dw1), want[4]["dw1"])
    assert moe.moe_device_status(d, b0.ws) == moe.MOE_OK
    with pytest.raises(moe.MoeError):  # the two sets must not share their inputs
        moe.moe_layer_steps_host(d, b0, b0, hx, hdy, hy, hdx)


@pytest.mark.parametrize("k", [3, 8, 12])
def test_fused_dispatch_bwd_matches_two_calls(k):
    """The layer path fuses the permute backward into the router's dx pass; it
    must give the same bits as moe_permute_bwd followed by moe_route_bwd."""
    inp = moe_synth.make_inputs(T=300, H=192, E=16, k=k, F=128, seed=30 + k)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    moe.moe_layer_forward(d, b)
    moe.moe_layer_backward(d, b, run_wgrad=False)
    dx32 = torch.empty_like(b.dx32)
    dx = torch.empty_like(b.dx)
    dw_r = torch.empty_like(b.dw_r)
    moe.moe_permute_bwd(d, b.dx_perm, b.slot, dx32)
    moe.moe_route_bwd(d, b.dgates, b.gates, b.idx, b.x, b.w_r, b.row_src, b.off, dx32, dx, dw_r,
                      b.ws)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert torch.equal(dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(dw_r.view(torch.int32), b.dw_r.view(torch.int32))
