"""GPU parity over seeded random layer shapes: the whole layer and each stage of
the CUDA path (through the C ABI) against the CPU oracle, as for the fixed
cases, on shapes drawn from a fixed seed so that combinations the named cases
do not cover (T, H, E, k, F, R and the routing mode together) get exercised,
including token counts that give each block of the fused dispatch several
tiles. Each shape is in the test's id, so a failure can be rerun by itself."""
import numpy as np
import pytest
import torch

import moe_synth

from _parity import check_stages, compare_layer, oracle_layer, run_layer

pytestmark = pytest.mark.gpu


def _shapes(n=12, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 5, 8, 12, 16, 24, 40, 64, 96, 128, 160, 256]))
        k = int(rng.integers(1, min(E, 16) + 1))
        divisors = [r for r in range(1, 9) if E % r == 0]
        R = int(rng.choice(divisors))
        T = int(rng.integers(1, 801))
        H = 64 * int(rng.integers(1, 13))
        F = 64 * int(rng.integers(1, 9))
        forced = rng.random() < 0.2
        bias = None if forced or E < 2 else rng.choice([None, "zipf_linear", "zipf_logrank"])
        out.append(dict(T=T, H=H, E=E, k=k, F=F, R=R,
                        mode=moe_synth.ROUTE_FORCED_BALANCED if forced
                        else moe_synth.ROUTE_SOFTMAX_TOPK,
                        bias=None if bias is None else str(bias), seed=100 + i))
    return out


def _shapes_many_tiles(n=6, seed=2027):
    """Token counts past one tile per block of the fused dispatch (147 blocks
    of 28 tokens), so blocks route, count and permute several tiles; small
    hidden sizes keep the oracle quick."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([8, 16, 32, 64, 96, 128]))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(4200, 12001))
        H = 64 * int(rng.integers(1, 5))
        F = 64 * int(rng.integers(1, 4))
        forced = rng.random() < 0.3
        bias = None if forced else rng.choice([None, "zipf_linear", "zipf_logrank"])
        out.append(dict(T=T, H=H, E=E, k=k, F=F, R=1,
                        mode=moe_synth.ROUTE_FORCED_BALANCED if forced
                        else moe_synth.ROUTE_SOFTMAX_TOPK,
                        bias=None if bias is None else str(bias), seed=200 + i))
    return out


SHAPES = _shapes() + _shapes_many_tiles()


def _id(s):
    return "T{T}-H{H}-E{E}-k{k}-F{F}-R{R}-m{mode}-{b}".format(b=s["bias"] or "nobias", **s)


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


@pytest.mark.parametrize("shape", SHAPES, ids=[_id(s) for s in SHAPES])
def test_random_shape_parity(shape):
    inp = moe_synth.make_inputs(**shape)
    g = run_layer(inp)
    o = oracle_layer(inp)
    ew = {}
    errs = compare_layer(g, o, elementwise=ew)
    stages = check_stages(g, inp)
    print(_id(shape), {k: f"{v:.2e}" for k, v in errs.items()})
    print(_id(shape), "element-wise", {k: f"{v:.2e}" for k, v in ew.items()})
    print(_id(shape), "stages", {k: {m: f"{x:.2e}" for m, x in v.items()} for k, v in stages.items()})
