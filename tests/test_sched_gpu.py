"""The two-stream, two-micro-batch scheduler: the overlapped schedule (with and
without the deferred wgrad) gives bit-identical results to the serial one, both
micro-batches match the oracle, and the phase timings describe real overlap."""
import numpy as np
import pytest
import torch

import combine_router_softmax_top_gb300 as moe
import moe_synth

from _parity import collect, compare_layer, desc_of, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


def make_pair(name=None, **kw):
    if name:
        i0, i1 = moe_synth.workload(name, 0), moe_synth.workload(name, 1)
    else:
        i0 = moe_synth.make_inputs(**kw, microbatch=0)
        i1 = moe_synth.make_inputs(**kw, microbatch=1)
    d = desc_of(i0)
    b0 = moe.LayerBuffers(d)
    b0.load_inputs(i0)
    b1 = moe.LayerBuffers(d, weights=b0)
    b1.load_inputs(i1, weights=False)
    return d, (i0, i1), (b0, b1)


def run(d, bufs, overlap, defer, steps=2, gemm_sms=0):
    sc = torch.cuda.Stream(priority=-1)
    sg = torch.cuda.Stream()
    torch.cuda.synchronize()
    s = moe.Scheduler(d, sc, sg, gemm_sms=gemm_sms)
    for _ in range(steps):
        s.step(bufs[0], bufs[1], overlap=overlap, defer_wgrad=defer)
    tm = s.timings()
    s.flush()
    torch.cuda.synchronize()
    for b in bufs:
        assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    s.close()
    return tm


SMALL = dict(T=384, H=256, E=16, k=4, F=256, seed=31, mode=moe_synth.ROUTE_FORCED_BALANCED)


def test_overlap_is_bit_identical_to_serial_and_matches_oracle():
    d, inps, bufs = make_pair(**SMALL)
    run(d, bufs, overlap=False, defer=False)
    ref = [collect(b, i) for b, i in zip(bufs, inps)]
    for overlap, defer in ((True, False), (True, True), (False, True), (2, False), (2, True)):
        for b in bufs:
            for n in ("y", "dx", "dw1", "dw2", "dw_r", "a", "h", "o", "da", "d_o"):
                getattr(b, n).zero_()
        run(d, bufs, overlap=overlap, defer=defer)
        got = [collect(b, i) for b, i in zip(bufs, inps)]
        for m in range(2):
            for key in ref[m]:
                assert np.array_equal(got[m][key], ref[m][key]), (overlap, defer, m, key)
    for m in range(2):
        compare_layer(ref[m], oracle_layer(inps[m]))


def test_timings_cover_every_phase_and_streams():
    d, inps, bufs = make_pair(**SMALL)
    tm = run(d, bufs, overlap=True, defer=True)
    phases = {(t["mb"], t["phase"]) for t in tm}
    for m in range(2):
        for p in ("dispatch", "ffn_fwd", "combine", "combine_bwd", "dgrad", "dispatch_bwd"):
            assert (m, p) in phases
    assert (0, "wgrad") in phases and (1, "wgrad") in phases  # the deferred one ran this step
    for t in tm:
        assert t["end_ms"] >= t["start_ms"] >= 0
        assert t["stream"] == (1 if t["phase"] in ("ffn_fwd", "dgrad", "wgrad") else 0)
    comm, gemm, hidden = moe.interval_overlap(tm)
    assert comm > 0 and gemm > 0 and hidden >= 0


def test_dispatch_only_overlap_timings():
    # overlap = 2: both dispatches on the comm stream first, the rest of each
    # micro-batch on the GEMM stream in layer order, each wgrad on the comm stream
    d, inps, bufs = make_pair(**SMALL)
    tm = run(d, bufs, overlap=2, defer=False, steps=1)
    assert len(tm) == 14
    for t in tm:
        on_comm = t["phase"] in ("dispatch", "wgrad")
        assert t["stream"] == (0 if on_comm else 1), t
    order = [(t["mb"], t["phase"]) for t in tm if t["stream"] == 1]
    assert order == [(m, p) for m in range(2) for p in
                     ("ffn_fwd", "combine", "combine_bwd", "dgrad", "dispatch_bwd")]
    start = {(t["mb"], t["phase"]): t["start_ms"] for t in tm}
    end = {(t["mb"], t["phase"]): t["end_ms"] for t in tm}
    for m in range(2):
        assert start[(m, "ffn_fwd")] >= end[(m, "dispatch")]
        assert start[(m, "wgrad")] >= end[(m, "dgrad")]


@pytest.mark.slow
@pytest.mark.parametrize("overlap", [True, 2])
def test_two_microbatch_workload_overlap_matches_serial(overlap):
    d, inps, bufs = make_pair("two_microbatch")
    run(d, bufs, overlap=False, defer=False, steps=1)
    ref = [collect(b, i) for b, i in zip(bufs, inps)]
    run(d, bufs, overlap=overlap, defer=True, steps=1)
    got = [collect(b, i) for b, i in zip(bufs, inps)]
    for m in range(2):
        for key in ref[m]:
            assert np.array_equal(got[m][key], ref[m][key]), (m, key)


@pytest.mark.parametrize("overlap,gemm_sms", [(True, 8), (True, 30), (True, 120), (2, 8),
                                              (2, 112), (2, 150)])
def test_capped_gemm_grid_is_bit_identical(overlap, gemm_sms):
    """With the GEMM grid capped, each CTA of a chained expert GEMM (FC1 -> FC2,
    FC2 dgrad -> FC1 dgrad) works through many rounds of tiles and the second
    GEMM's tiles wait on other CTAs' first-GEMM tiles; under overlap = 2 the cap
    splits the GPU between expert forward 0 and dispatch 1, whose blocks then
    take several token tiles each. Same bits as uncapped."""
    d, inps, bufs = make_pair(**SMALL)
    run(d, bufs, overlap=False, defer=False)
    ref = [collect(b, i) for b, i in zip(bufs, inps)]
    for b in bufs:
        for n in ("y", "dx", "dw1", "dw2", "dw_r", "a", "h", "o", "da", "d_o", "dx_perm"):
            getattr(b, n).zero_()
    run(d, bufs, overlap=overlap, defer=True, gemm_sms=gemm_sms)
    got = [collect(b, i) for b, i in zip(bufs, inps)]
    for m in range(2):
        for key in ref[m]:
            assert np.array_equal(got[m][key], ref[m][key]), (overlap, gemm_sms, m, key)
