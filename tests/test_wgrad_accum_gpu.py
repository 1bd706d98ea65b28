"""Gradient accumulation fusion on the GPU: the expert weight gradients added
into fp32 main gradients by the wgrad GEMM's epilogue (TMA reductions), against
the oracle's accumulation, through the entry point, the layer path and the
two-stream scheduler."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth
from oracle import moe_oracle as O

from _parity import assert_close, desc_of, np64, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


def dev(a, dt):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dt).cuda()


def rand_main(shape, scale, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * scale)


CASES = {
    # ragged rows per expert, empty experts, partial tiles in every dimension
    "ragged_empty": lambda: moe_synth.make_inputs(T=300, H=192, E=16, k=2, F=192, seed=41,
                                                  bias="zipf_logrank"),
    # several 128-row M blocks and 256-column N blocks per expert
    "multi_tile": lambda: moe_synth.make_inputs(T=1000, H=320, E=8, k=4, F=448, seed=42),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_entry_point_matches_oracle(case):
    """Two calls on a random main gradient: each adds the expert gradient once."""
    inp = CASES[case]()
    o = oracle_layer(inp)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    E, H, F = inp.E, inp.H, inp.F
    scale1 = float(np.abs(o["dw1"]).max())
    scale2 = float(np.abs(o["dw2"]).max())
    m1 = rand_main((E, 2 * F, H), scale1, 1)
    m2 = rand_main((E, H, F), scale2, 2)
    gm1, gm2 = m1.cuda(), m2.cuda()
    x_perm, h = dev(o["x_perm"], torch.bfloat16), dev(o["h"], torch.bfloat16)
    d_o, da = dev(o["d_o"], torch.bfloat16), dev(o["da"], torch.bfloat16)
    off = dev(o["off"], torch.int32)
    args = (o["x_perm"], o["h"], o["d_o"], o["da"], o["off"], E)
    want1, want2 = m1.numpy(), m2.numpy()
    for call in range(2):
        moe.moe_expert_ffn_bwd_wgrad_accum(d, x_perm, h, d_o, da, off, gm1, gm2, b.ws)
        want1, want2 = O.expert_ffn_bwd_wgrad_accum(want1, want2, *args)
        got1, got2 = gm1.cpu().numpy(), gm2.cpu().numpy()
        # the increment, against the oracle's, scaled by the gradient's size
        assert_close(f"dw1 step {call}", got1.astype(np.float64) - m1.numpy(),
                     want1.astype(np.float64) - m1.numpy(), tol=1e-3)
        assert_close(f"dw2 step {call}", got2.astype(np.float64) - m2.numpy(),
                     want2.astype(np.float64) - m2.numpy(), tol=1e-3)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    # experts with no rows are left exactly as they were
    cnt = np.diff(o["off"])
    for e in np.flatnonzero(cnt == 0):
        assert torch.equal(gm1[e].cpu(), m1[e]) and torch.equal(gm2[e].cpu(), m2[e]), e


def test_accumulating_from_zero_gives_the_stored_gradient_bits():
    """From a zero main gradient the fp32 sum is the accumulator itself, so its
    bf16 rounding equals the overwriting wgrad's output bit for bit."""
    inp = CASES["multi_tile"]()
    o = oracle_layer(inp)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    E, H, F = inp.E, inp.H, inp.F
    x_perm, h = dev(o["x_perm"], torch.bfloat16), dev(o["h"], torch.bfloat16)
    d_o, da = dev(o["d_o"], torch.bfloat16), dev(o["da"], torch.bfloat16)
    off = dev(o["off"], torch.int32)
    gm1 = torch.zeros(E, 2 * F, H, device="cuda")
    gm2 = torch.zeros(E, H, F, device="cuda")
    moe.moe_expert_ffn_bwd_wgrad_accum(d, x_perm, h, d_o, da, off, gm1, gm2, b.ws)
    moe.moe_expert_ffn_bwd_wgrad(d, x_perm, h, d_o, da, off, b.dw1, b.dw2, b.ws)
    assert torch.equal(gm1.to(torch.bfloat16).float(), b.dw1.float())
    assert torch.equal(gm2.to(torch.bfloat16).float(), b.dw2.float())


def test_layer_path_accumulates_two_micro_batches():
    """Forward + backward of two micro-batches with MOE_FLAG_WGRAD_ACCUM_FP32 into
    one main gradient: the oracle's two accumulations, in call order."""
    inps = [moe_synth.make_inputs(T=256, H=256, E=8, k=2, F=256, seed=43, microbatch=m)
            for m in range(2)]
    d = desc_of(inps[0])
    d.flags = moe.FLAG_WGRAD_ACCUM_FP32
    b = moe.LayerBuffers(d)
    assert b.dw1 is None and b.main_dw1 is not None
    E, H, F = inps[0].E, inps[0].H, inps[0].F
    m1 = rand_main((E, 2 * F, H), 1e-2, 3)
    m2 = rand_main((E, H, F), 1e-2, 4)
    b.main_dw1.copy_(m1)
    b.main_dw2.copy_(m2)
    want1, want2 = m1.numpy(), m2.numpy()
    for i, inp in enumerate(inps):
        b.load_inputs(inp, weights=(i == 0))
        moe.moe_layer_forward(d, b)
        moe.moe_layer_backward(d, b)
        o = oracle_layer(inp)
        want1, want2 = O.expert_ffn_bwd_wgrad_accum(want1, want2, o["x_perm"], o["h"],
                                                    o["d_o"], o["da"], o["off"], E)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert_close("main_dw1", np64(b.main_dw1) - m1.numpy(), want1.astype(np.float64) - m1.numpy())
    assert_close("main_dw2", np64(b.main_dw2) - m2.numpy(), want2.astype(np.float64) - m2.numpy())


def test_scheduler_accumulation_is_bit_identical_to_serial():
    kw = dict(T=384, H=256, E=16, k=4, F=256, seed=44, mode=moe_synth.ROUTE_FORCED_BALANCED)
    results = []
    for overlap, defer in ((False, False), (True, False), (True, True)):
        i0 = moe_synth.make_inputs(**kw, microbatch=0)
        i1 = moe_synth.make_inputs(**kw, microbatch=1)
        d = desc_of(i0)
        d.flags = moe.FLAG_WGRAD_ACCUM_FP32
        b0 = moe.LayerBuffers(d)
        b0.load_inputs(i0)
        b1 = moe.LayerBuffers(d, weights=b0)
        b1.load_inputs(i1, weights=False)
        sc, sg = torch.cuda.Stream(priority=-1), torch.cuda.Stream()
        torch.cuda.synchronize()
        s = moe.Scheduler(d, sc, sg)
        for _ in range(2):
            s.step(b0, b1, overlap=overlap, defer_wgrad=defer)
        s.flush()
        torch.cuda.synchronize()
        for b in (b0, b1):
            assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
        s.close()
        results.append([t.cpu() for t in (b0.main_dw1, b0.main_dw2, b1.main_dw1, b1.main_dw2)])
    for other in results[1:]:
        for a, b in zip(results[0], other):
            assert torch.equal(a, b)
    # two steps of the same micro-batch: twice the oracle's gradient
    o = oracle_layer(i0)
    z1, z2 = O.expert_ffn_bwd_wgrad_accum(np.zeros(tuple(b0.main_dw1.shape), np.float32),
                                          np.zeros(tuple(b0.main_dw2.shape), np.float32),
                                          o["x_perm"], o["h"], o["d_o"], o["da"], o["off"],
                                          i0.E)
    assert_close("mb0 main_dw1", results[0][0].double().numpy(), 2.0 * z1.astype(np.float64))
    assert_close("mb0 main_dw2", results[0][1].double().numpy(), 2.0 * z2.astype(np.float64))


def test_zero_tokens_leave_main_gradients_alone():
    inp = moe_synth.make_inputs(T=0, H=128, E=8, k=2, F=128, seed=45)
    d = desc_of(inp)
    d.flags = moe.FLAG_WGRAD_ACCUM_FP32
    b = moe.LayerBuffers(d)
    b.main_dw1.fill_(1.5)
    b.main_dw2.fill_(-2.5)
    moe.moe_layer_forward(d, b)
    moe.moe_layer_backward(d, b)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert float(b.main_dw1.min()) == 1.5 == float(b.main_dw1.max())
    assert float(b.main_dw2.min()) == -2.5 == float(b.main_dw2.max())
