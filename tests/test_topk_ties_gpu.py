"""Top-k routing where logits tie exactly: duplicated router rows, all-zero
rows, tokens whose logits are all zero, and experts masked by a -inf bias.
The GPU's choice (descending logit, ties to the lower expert index) must give
the oracle's indices bit for bit, through the fused router (E <= 128) and the
separate top-k kernel (E > 128), alone and inside the fused dispatch."""
import numpy as np
import pytest
import torch

import moe_synth
from oracle import moe_oracle as O

from _parity import desc_of, npi, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_softmax_top_gb300 import build
    build.build()
    torch.cuda.init()


def _tied_inputs(T, H, E, k, seed):
    inp = moe_synth.make_inputs(T=T, H=H, E=E, k=k, F=64, seed=seed,
                                mode=moe_synth.ROUTE_SOFTMAX_TOPK)
    w = inp.w_r.clone()
    w[5] = w[5] * 4  # a power of two: exact in bf16, and often in the top k
    w[9] = w[5]
    w[20] = w[5]      # experts 5, 9, 20 tie on every token
    w[3] = w[2]       # 2 and 3 tie
    w[11] = 0
    w[12] = 0         # logit exactly 0 for both, on every token
    inp.w_r = w
    x = inp.x.clone()
    x[0] = 0          # token 0: every logit 0, so the k lowest experts win
    x[7] = 0
    inp.x = x
    bias = torch.zeros(E, dtype=torch.float32)
    bias[E - 1] = float("-inf")
    bias[E - 2] = float("-inf")  # never chosen while k < E - 2
    inp.bias = bias
    return inp


def _oracle_route(inp):
    z = O.router_logits_fp32(inp.x.float().numpy(), inp.w_r.float().numpy(),
                             inp.bias.numpy())
    return O.route_topk(z, inp.k)


@pytest.mark.parametrize("E,k", [(32, 6), (128, 8), (160, 8)])
def test_route_ties_match_the_oracle(E, k):
    import combine_router_softmax_top_gb300 as moe
    inp = _tied_inputs(T=300, H=128, E=E, k=k, seed=71)
    idx_o, gates_o = _oracle_route(inp)
    assert list(idx_o[0]) == list(range(k))  # the all-zero token
    assert not np.isin([E - 1, E - 2], idx_o).any()
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    moe.moe_route(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.ws)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert np.array_equal(npi(b.idx), idx_o)
    assert np.max(np.abs(np64(b.gates) - gates_o)) < 1e-5


def test_fused_dispatch_ties_match_the_oracle():
    import combine_router_softmax_top_gb300 as moe
    inp = _tied_inputs(T=500, H=128, E=64, k=8, seed=72)
    idx_o, gates_o = _oracle_route(inp)
    d = desc_of(inp)
    b = moe.LayerBuffers(d)
    b.load_inputs(inp)
    moe.moe_dispatch_fused(d, b.x, b.w_r, b.bias, b.logits, b.idx, b.gates, b.cnt, b.off,
                           b.slot, b.row_src, b.cnt_re, b.rank_off, b.x_perm, b.ws)
    assert moe.moe_device_status(d, b.ws) == moe.MOE_OK
    assert np.array_equal(npi(b.idx), idx_o)
    assert np.max(np.abs(np64(b.gates) - gates_o)) < 1e-5
    lay = O.dispatch_layout(idx_o, inp.E, inp.R)
    for key in ("cnt", "off", "slot", "row_src"):
        got = npi(getattr(b, key))
        assert np.array_equal(got[: len(lay[key])].reshape(np.shape(lay[key])), lay[key]), key
