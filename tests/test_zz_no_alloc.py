"""The allocation-free dispatch layout (moe_dispatch_layout_static).

It serves callers that cannot hand the library a workspace, such as a plugin
that only receives its input and output tensors, or code being captured into a
CUDA graph where cudaMalloc is not allowed. It must give exactly the layout of
the workspace-based moe_dispatch_layout (integer outputs, so bit for bit) on
two calls in a row with different routings, since its scratch array is shared
and keeps the previous call's contents. This file is collected last.
"""
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth

pytestmark = pytest.mark.gpu

OUTS = ("cnt", "off", "slot", "row_src", "cnt_re", "rank_off")


def layouts(d, idx):
    ref = moe.LayerBuffers(d)
    got = moe.LayerBuffers(d)
    for b in (ref, got):
        for n in OUTS:
            getattr(b, n).fill_(-7)
    moe.moe_dispatch_layout(d, idx, ref.cnt, ref.off, ref.slot, ref.row_src, ref.cnt_re,
                            ref.rank_off, ref.ws)
    moe.moe_dispatch_layout_static(d, idx, got.cnt, got.off, got.slot, got.row_src, got.cnt_re,
                                   got.rank_off)
    torch.cuda.synchronize()
    return ref, got


def test_static_layout_matches_workspace_layout_on_two_calls():
    from combine_router_softmax_top_gb300 import build
    build.build()
    # two different routings back to back: skewed (empty experts), then balanced
    inp1 = moe_synth.make_inputs(T=3000, H=256, E=64, k=8, F=64, R=8, seed=41,
                                 bias="zipf_logrank")
    inp2 = moe_synth.make_inputs(T=1000, H=256, E=64, k=8, F=64, R=8, seed=42,
                                 mode=moe_synth.ROUTE_FORCED_BALANCED)
    for inp in (inp1, inp2):
        d = moe.LayerDesc.of(**inp.shape_dict())
        b = moe.LayerBuffers(d)
        b.load_inputs(inp)
        moe.moe_route(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.ws)
        ref, got = layouts(d, b.idx)
        for n in OUTS:
            assert torch.equal(getattr(ref, n), getattr(got, n)), n


def test_static_layout_at_its_size_limit():
    """T = 65536 tokens and E = 256 experts fill the scratch array exactly."""
    inp = moe_synth.make_inputs(T=65536, H=64, E=256, k=1, F=64, R=4, seed=43)
    d = moe.LayerDesc.of(**inp.shape_dict())
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    moe.moe_route(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.ws)
    ref, got = layouts(d, b.idx)
    for n in OUTS:
        assert torch.equal(getattr(ref, n), getattr(got, n)), n
    assert moe.moe_dispatch_layout_static_status() == moe.MOE_OK


def test_static_layout_skips_and_reports_out_of_range_ids():
    """Ids E and -1: slot is -1 there, the other outputs equal the workspace
    path's bit for bit, and both paths report the skipped entries."""
    T, E, k = 700, 16, 3
    d = moe.LayerDesc.of(T=T, H=64, E=E, k=k, F=64, R=2)
    g = torch.Generator().manual_seed(44)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    idx[5, 1] = E
    idx[300, 0] = -1
    idx[699, 2] = E + 7
    idx = idx.cuda()
    ref, got = layouts(d, idx)
    assert moe.moe_device_status(d, ref.ws) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_dispatch_layout_static_status() == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_dispatch_layout_static_status() == moe.MOE_OK  # cleared by the read
    for n in OUTS:
        assert torch.equal(getattr(ref, n), getattr(got, n)), n
    for t, j in ((5, 1), (300, 0), (699, 2)):
        assert int(got.slot[t, j]) == -1
    assert int(got.off[E]) == T * k - 3
    # a clean call after it reports nothing
    fixed = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    layouts(d, fixed.cuda())
    assert moe.moe_dispatch_layout_static_status() == moe.MOE_OK


def test_static_layout_rejects_shapes_beyond_its_scratch():
    d = moe.LayerDesc.of(T=65537, H=128, E=8, k=1, F=64)
    idx = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_layout_static(d, idx, idx, idx, idx, idx, idx, idx)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
