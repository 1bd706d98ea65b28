"""CUDA-graph capture of the layer (moe_graph_capture): a replay matches the
oracle on every output of its scope, gives the same bits as the eager calls on
the same inputs, reads its buffers afresh on every replay, keeps the
side-stream fork/join and the accumulation flag, and rejects what cannot be
captured."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth
from oracle import moe_oracle as O

from _parity import FLOAT_KEYS, INT_KEYS, assert_close, collect, compare_layer, desc_of, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


OUTS = {
    moe.GRAPH_ROUTER_PREPROCESS: ("logits", "idx", "gates", "cnt", "off", "slot", "row_src",
                                  "cnt_re", "rank_off", "x_perm"),
}
OUTS[moe.GRAPH_LAYER_FORWARD] = OUTS[moe.GRAPH_ROUTER_PREPROCESS] + ("a", "h", "o", "y")
OUTS[moe.GRAPH_LAYER_STEP] = OUTS[moe.GRAPH_LAYER_FORWARD] + (
    "d_o", "dgates", "da", "dx_perm", "dx", "dw_r", "dw1", "dw2")


def eager(scope, d, b, st):
    with torch.cuda.stream(st):
        if scope == moe.GRAPH_ROUTER_PREPROCESS:
            moe.moe_route(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.ws, st)
            moe.moe_dispatch_layout(d, b.idx, b.cnt, b.off, b.slot, b.row_src, b.cnt_re,
                                    b.rank_off, b.ws, st)
            moe.moe_permute(d, b.x, b.row_src, b.x_perm, st)
        else:
            moe.moe_layer_forward(d, b, st)
            if scope == moe.GRAPH_LAYER_STEP:
                moe.moe_layer_backward(d, b, True, st)


def same_bits(b1, b2, names):
    for n in names:
        t1, t2 = getattr(b1, n), getattr(b2, n)
        if t1 is None:
            assert t2 is None, n
            continue
        assert torch.equal(t1.view(torch.uint8), t2.view(torch.uint8)), n


CASE = dict(T=600, H=256, E=16, k=4, F=256, R=2, seed=51)

# outputs of each scope in the oracle's names (logits is compared bit for bit)
SCOPE_KEYS = {
    moe.GRAPH_ROUTER_PREPROCESS: set(INT_KEYS) | {"logits", "gates", "x_perm"},
}
SCOPE_KEYS[moe.GRAPH_LAYER_FORWARD] = SCOPE_KEYS[moe.GRAPH_ROUTER_PREPROCESS] | {"a", "h", "o",
                                                                                 "y"}
SCOPE_KEYS[moe.GRAPH_LAYER_STEP] = SCOPE_KEYS[moe.GRAPH_LAYER_FORWARD] | {
    "d_o", "dgates", "da", "dx_perm", "dx", "dw_r", "dw1", "dw2"}


@pytest.mark.parametrize("scope,flags", [(moe.GRAPH_ROUTER_PREPROCESS, 0),
                                         (moe.GRAPH_LAYER_FORWARD, 0),
                                         (moe.GRAPH_LAYER_STEP, 0),
                                         (moe.GRAPH_LAYER_STEP, moe.FLAG_WGRAD_ACCUM_FP32)])
def test_replay_matches_oracle(scope, flags):
    """Each replay of a captured scope, on new inputs copied into the captured
    buffers, against the oracle of those inputs: integers and logits exact,
    floats within 2e-2. Under MOE_FLAG_WGRAD_ACCUM_FP32 the main gradients
    start at zero and take one accumulation per replay."""
    st = torch.cuda.Stream()
    inps = [moe_synth.make_inputs(**CASE, microbatch=m) for m in range(2)]
    d = desc_of(inps[0])
    d.flags = flags
    b = moe.LayerBuffers(d)
    b.load_inputs(inps[0])
    torch.cuda.synchronize()
    g = moe.Graph(d, b, scope, st)
    keys = SCOPE_KEYS[scope]
    if flags:
        keys = keys - {"dw1", "dw2"}
    skip = (set(INT_KEYS) | set(FLOAT_KEYS) | {"logits"}) - keys
    for inp in inps:
        b.x.copy_(inp.x)
        b.dy.copy_(inp.dy)
        if flags:
            b.main_dw1.zero_()
            b.main_dw2.zero_()
        torch.cuda.synchronize()
        g.replay(st)
        st.synchronize()
        assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
        got = collect(b, inp)
        ora = oracle_layer(inp)
        errs = compare_layer(got, ora, skip=skip)
        print(scope, flags, {k: f"{v:.2e}" for k, v in errs.items()})
        if flags:
            z1 = np.zeros(tuple(inp.w1.shape), np.float32)
            z2 = np.zeros(tuple(inp.w2.shape), np.float32)
            m1, m2 = O.expert_ffn_bwd_wgrad_accum(z1, z2, ora["x_perm"], ora["h"], ora["d_o"],
                                                  ora["da"], ora["off"], inp.E)
            assert_close("main_dw1", got["main_dw1"], m1)
            assert_close("main_dw2", got["main_dw2"], m2)
    g.close()


@pytest.mark.parametrize("scope", [moe.GRAPH_ROUTER_PREPROCESS, moe.GRAPH_LAYER_FORWARD,
                                   moe.GRAPH_LAYER_STEP])
def test_replay_matches_eager_and_rereads_inputs(scope):
    st = torch.cuda.Stream()
    inps = [moe_synth.make_inputs(**CASE, microbatch=m) for m in range(2)]
    d = desc_of(inps[0])
    bg = moe.LayerBuffers(d)
    bg.load_inputs(inps[0])
    torch.cuda.synchronize()
    g = moe.Graph(d, bg, scope, st)
    assert g.kernels >= 1
    for inp in inps:  # the second replay sees new x and dy in the same buffers
        be = moe.LayerBuffers(d)
        be.load_inputs(inp)
        bg.x.copy_(inp.x)
        bg.dy.copy_(inp.dy)
        torch.cuda.synchronize()
        eager(scope, d, be, st)
        l0 = moe.moe_kernel_launches()
        g.replay(st)
        assert moe.moe_kernel_launches() - l0 == g.kernels
        st.synchronize()
        assert moe.moe_device_status(d, bg.ws) == moe.MOE_OK
        same_bits(be, bg, OUTS[scope])
    g.close()


def test_step_graph_with_fp32_accumulation_matches_eager_steps():
    st = torch.cuda.Stream()
    inp = moe_synth.make_inputs(T=256, H=128, E=8, k=2, F=128, seed=52)
    d = desc_of(inp)
    d.flags = moe.FLAG_WGRAD_ACCUM_FP32
    be, bg = moe.LayerBuffers(d), moe.LayerBuffers(d)
    be.load_inputs(inp)
    bg.load_inputs(inp)
    torch.cuda.synchronize()
    g = moe.Graph(d, bg, moe.GRAPH_LAYER_STEP, st)
    for _ in range(3):
        eager(moe.GRAPH_LAYER_STEP, d, be, st)
        g.replay(st)
    st.synchronize()
    same_bits(be, bg, ("main_dw1", "main_dw2", "dx", "dw_r"))
    assert float(bg.main_dw1.abs().max()) > 0
    g.close()


def test_capture_is_refused_where_it_cannot_work():
    inp = moe_synth.make_inputs(T=64, H=128, E=8, k=2, F=128, seed=53)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    st = torch.cuda.Stream()
    with pytest.raises(moe.MoeError) as e:
        moe.Graph(d, b, moe.GRAPH_LAYER_FORWARD, 0)  # the legacy default stream
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.Graph(d, b, 7, st)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    moe.moe_profile_start(64)
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.Graph(d, b, moe.GRAPH_LAYER_FORWARD, st)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_profile_stop(64)
    # nothing was left capturing: eager work on the stream still runs
    eager(moe.GRAPH_LAYER_FORWARD, d, b, st)
    st.synchronize()
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
