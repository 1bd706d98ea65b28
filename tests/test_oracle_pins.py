"""Pins of the CPU oracle to facts outside itself.

Each test checks the oracle against something it does not compute the same way:
closed forms, brute force on tiny inputs, invariants of the dispatch layout,
special cases that reduce to a dense textbook SwiGLU FFN (evaluated with torch
library routines), and float64 central finite differences of the whole layer.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_synth
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_inputs(T=24, H=16, E=6, k=3, F=8, R=1, mode=0, seed=7, bias=None,
                 x_std=1.0, w_std=0.3):
    return moe_synth.make_inputs(T=T, H=H, E=E, k=k, F=F, R=R, mode=mode, bias=bias,
                                 seed=seed, x_std=x_std, w_std=w_std)


# ----------------------------------------------------------------------------- rounding
def test_bf16_rne_hand_cases():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 spacing just above 1
    cases = {
        one + ulp / 2: one,              # tie -> even (mantissa 0)
        one + 3 * ulp / 2: one + 2 * ulp,  # tie -> even (mantissa 2)
        one + ulp / 2 + 2.0 ** -30: one + ulp,  # just above the tie -> up
        -(one + ulp / 2): -one,
        0.0: 0.0,
        3.0: 3.0,
    }
    for v, want in cases.items():
        assert O.bf16_rne(np.array([v]))[0] == want, v


def test_bf16_rne_matches_torch_on_fp32_values():
    # torch rounds float32 -> bfloat16 to nearest even in one step; on values that
    # are exact in float32 the oracle's float64 rounding must agree bit for bit.
    g = np.random.default_rng(3)
    a = g.standard_normal(200000).astype(np.float32) * np.float32(10.0)
    bits = a.view(np.uint32)
    ties = (bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)  # exact halfway cases
    a = np.concatenate([a, ties.view(np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_rne(a.astype(np.float64))
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------- router
def test_logits_integer_closed_form():
    # small integers: every partial sum is exact, so z must equal the integer dot product
    g = np.random.default_rng(0)
    x = g.integers(-4, 5, size=(9, 33)).astype(np.float64)
    w = g.integers(-3, 4, size=(5, 33)).astype(np.float64)
    want = np.einsum("th,eh->te", x.astype(np.int64), w.astype(np.int64))
    assert np.array_equal(O.router_logits_fp32(x, w), want.astype(np.float32))
    b = np.array([0.5, -1.0, 2.0, 0.0, 0.25])
    assert np.array_equal(O.router_logits_fp32(x, w, b), (want + b).astype(np.float32))


def test_logits_within_recursive_summation_bound():
    inp = small_inputs(T=64, H=256, E=16, w_std=0.05)
    x, w = O._np(inp.x), O._np(inp.w_r)
    z = O.router_logits_fp32(x, w).astype(np.float64)
    exact = x @ w.T
    u = 2.0 ** -24
    H = x.shape[1]
    bound = (H - 1) * u / (1 - (H - 1) * u) * (np.abs(x) @ np.abs(w).T)
    assert np.all(np.abs(z - exact) <= bound)


def test_topk_against_subset_brute_force():
    inp = small_inputs(T=40, H=16, E=6, k=3, seed=11)
    z = O.router_logits_fp32(O._np(inp.x), O._np(inp.w_r))
    idx, gates = O.route_topk(z, 3)
    for t in range(z.shape[0]):
        best = max(itertools.combinations(range(6), 3),
                   key=lambda s: (sum(float(z[t, e]) for e in s), [-e for e in s]))
        assert set(idx[t].tolist()) == set(best)
        # slot order: descending logit
        assert all(z[t, idx[t, j]] >= z[t, idx[t, j + 1]] for j in range(2))


def test_topk_ties_go_to_lower_expert():
    z = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]], dtype=np.float32)
    idx, _ = O.route_topk(z, 2)
    assert idx.tolist() == [[1, 2]]
    idx, _ = O.route_topk(z, 4)
    assert idx.tolist() == [[1, 2, 4, 0]]


def test_gates_equal_softmax_of_selected_logits():
    import scipy.special
    inp = small_inputs(T=50, E=8, k=3, seed=5)
    z = O.router_logits_fp32(O._np(inp.x), O._np(inp.w_r))
    idx, gates = O.route_topk(z, 3)
    want = scipy.special.softmax(np.take_along_axis(z.astype(np.float64), idx, 1), axis=1)
    np.testing.assert_allclose(gates, want, rtol=1e-12, atol=0)
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=1e-14)


def test_forced_routing_closed_form_and_balance():
    T, E, k = 4096, 128, 8
    z = np.zeros((T, E), np.float32)
    idx, gates = O.route_forced(z, k)
    t = np.arange(T)[:, None]
    assert np.array_equal(idx, (8 * t + np.arange(8)[None]) % 128)
    np.testing.assert_allclose(gates, 1.0 / k)  # equal logits -> equal gates
    lay = O.dispatch_layout(idx, E)
    assert np.all(lay["cnt"] == T * k // E)


# ----------------------------------------------------------------------------- worked example
def test_worked_example():
    """Hand-derived routing of three tokens over four experts (values in the fixture)."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    x = np.array(ex["x"], np.float64)
    w = np.array(ex["w_r"], np.float64)
    z = O.router_logits_fp32(x, w)
    assert z.tolist() == ex["logits"]
    idx, gates = O.route_topk(z, ex["k"])
    assert idx.tolist() == ex["idx"]
    e = math.e
    want_gates = [[e / (e + 1), 1 / (e + 1)], [0.5, 0.5], [e * e / (e * e + 1), 1 / (e * e + 1)]]
    np.testing.assert_allclose(gates, want_gates, rtol=1e-15)
    lay = O.dispatch_layout(idx, ex["E"], ex["R"])
    for key in ("cnt", "off", "slot", "row_src", "cnt_re", "rank_off"):
        assert np.asarray(lay[key]).tolist() == ex[key], key
    fidx, fg = O.route_forced(z, ex["k"])
    assert fidx.tolist() == ex["forced_idx"]
    want_fg = [[e / (e + 1), 1 / (e + 1)], [e * e / (e * e + 1), 1 / (e * e + 1)], [0.5, 0.5]]
    np.testing.assert_allclose(fg, want_fg, rtol=1e-15)
    # router backward for dgates = [1, 0] on token 0: dz_S = [g0 g1, -g0 g1]
    dg = np.zeros((3, 2))
    dg[0, 0] = 1.0
    dz, _, _ = O.route_bwd(dg, z, idx, x, w, np.zeros((3, 2)), rnd=O.identity)
    g0g1 = e / (e + 1) ** 2
    want_dz = np.zeros((3, 4))
    want_dz[0, 2], want_dz[0, 0] = g0g1, -g0g1
    np.testing.assert_allclose(dz, want_dz, atol=1e-15)


# ----------------------------------------------------------------------------- layout
def brute_force_slots(idx, E):
    """Scan experts in order, then tokens in order: the definition of the stable layout."""
    T, k = idx.shape
    slot = -np.ones((T, k), np.int64)
    nxt = 0
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    slot[t, j] = nxt
                    nxt += 1
    return slot


@pytest.mark.parametrize("T,E,k,R,mode", [(37, 8, 2, 1, 0), (64, 16, 4, 4, 0), (33, 6, 6, 3, 0),
                                          (50, 5, 1, 1, 0), (40, 12, 3, 2, 1)])
def test_layout_brute_force_and_invariants(T, E, k, R, mode):
    inp = small_inputs(T=T, E=E, k=k, R=R, mode=mode, seed=T + E)
    z = O.router_logits_fp32(O._np(inp.x), O._np(inp.w_r))
    idx, _ = (O.route_forced if mode else O.route_topk)(z, k)
    lay = O.dispatch_layout(idx, E, R)
    assert np.array_equal(lay["slot"], brute_force_slots(idx, E))
    N = T * k
    assert lay["cnt"].sum() == N and lay["off"][-1] == N
    assert np.all(np.diff(lay["off"]) == lay["cnt"])
    # slot and row_src are inverse permutations of 0..N-1
    assert np.array_equal(np.sort(lay["row_src"]), np.arange(N))
    assert np.array_equal(lay["row_src"][lay["slot"].reshape(-1)], np.arange(N))
    # every token appears exactly k times; rows of an expert ascend by token
    assert np.all(np.bincount(lay["row_src"] // k, minlength=T) == k)
    for e in range(E):
        toks = lay["row_src"][lay["off"][e]:lay["off"][e + 1]] // k
        assert np.all(np.diff(toks) > 0)
        assert np.all(idx.reshape(-1)[lay["row_src"][lay["off"][e]:lay["off"][e + 1]]] == e)
    # per-rank tables: the send buffer is rank-major
    E_l = E // R
    assert lay["cnt_re"].shape == (R, E_l)
    assert np.array_equal(np.diff(lay["rank_off"]), lay["cnt_re"].sum(1))
    for s in range(N):
        e = idx.reshape(-1)[lay["row_src"][s]]
        r = e // E_l
        assert lay["rank_off"][r] <= s < lay["rank_off"][r + 1]


# ----------------------------------------------------------------------------- dispatch/combine
def test_combine_of_dispatch_is_identity():
    inp = small_inputs(T=30, H=16, E=5, k=2, seed=3)
    x = O._np(inp.x)
    z = O.router_logits_fp32(x, O._np(inp.w_r))
    idx, gates = O.route_topk(z, 2)
    lay = O.dispatch_layout(idx, 5)
    xp = O.permute(x, lay["row_src"], 2)
    y = O.combine(xp, lay["slot"], gates, rnd=O.identity)   # identity experts: o = x_perm
    np.testing.assert_allclose(y, x, rtol=1e-14, atol=1e-14)
    y16 = O.combine(xp, lay["slot"], gates)                 # one bf16 rounding at the end
    assert np.array_equal(y16, x)


def _dense_swiglu(x, w1, w2):
    """Dense SwiGLU FFN from torch library routines (textbook form)."""
    xt = torch.as_tensor(x, dtype=torch.float64)
    a = xt @ torch.as_tensor(w1, dtype=torch.float64).T
    F = a.shape[1] // 2
    h = torch.nn.functional.silu(a[:, :F]) * a[:, F:]
    return (h @ torch.as_tensor(w2, dtype=torch.float64).T).numpy()


def test_single_expert_reduces_to_dense_ffn():
    inp = small_inputs(T=20, H=16, E=1, k=1, F=8, seed=2)
    fwd = O.layer_forward(inp, rnd=O.identity)
    np.testing.assert_allclose(fwd["gates"], 1.0)
    want = _dense_swiglu(O._np(inp.x), O._np(inp.w1)[0], O._np(inp.w2)[0])
    np.testing.assert_allclose(fwd["y"], want, rtol=1e-12, atol=1e-12)


def test_identical_experts_reduce_to_dense_ffn():
    inp = small_inputs(T=25, H=16, E=4, k=2, F=8, seed=9)
    inp.w1 = inp.w1[:1].repeat(4, 1, 1)
    inp.w2 = inp.w2[:1].repeat(4, 1, 1)
    fwd = O.layer_forward(inp, rnd=O.identity)
    want = _dense_swiglu(O._np(inp.x), O._np(inp.w1)[0], O._np(inp.w2)[0])
    np.testing.assert_allclose(fwd["y"], want, rtol=1e-12, atol=1e-12)


def test_swiglu_and_its_gradient_against_torch_over_both_tails():
    """SwiGLU and its gradient against torch's silu and autograd in float64, on
    pre-activations far into both tails of the sigmoid (|a_gate| up to 40),
    element by element: the large-|gate| regime the GPU epilogue must also
    handle without losing the sigmoid's relative accuracy."""
    g = np.random.default_rng(17)
    rows, F = 64, 48
    ag = np.concatenate([np.linspace(-40.0, 40.0, rows * F // 2),
                         g.standard_normal(rows * F // 2) * 8.0]).reshape(rows, F)
    au = g.standard_normal((rows, F)) * 3.0
    a = np.concatenate([ag, au], axis=1)
    dh = g.standard_normal((rows, F))
    at = torch.tensor(a, dtype=torch.float64, requires_grad=True)
    ht = torch.nn.functional.silu(at[:, :F]) * at[:, F:]
    ht.backward(torch.tensor(dh))
    want_h, want_da = ht.detach().numpy(), at.grad.numpy()
    np.testing.assert_allclose(O.swiglu(a, O.identity), want_h, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(O.swiglu_bwd(dh, a, O.identity), want_da, rtol=1e-11,
                               atol=1e-300)
    # with the bf16 rounding of R8: one rounding of those values
    assert np.array_equal(O.swiglu(a), O.bf16_rne(O.swiglu(a, O.identity)))
    # deep negative gates: silu(u) ~ u e^u, nonzero and of the right sign
    h = O.swiglu(a, O.identity)
    deep = ag < -20
    assert np.all(np.sign(h[deep]) == -np.sign(au[deep]))


# ----------------------------------------------------------------------------- gradients
def _loss(inp, dy):
    fwd = O.layer_forward(inp, rnd=O.identity, exact_logits=True)
    return float((fwd["y"] * dy).sum()), fwd["idx"]


@pytest.mark.parametrize("mode", [0, 1])
def test_gradients_against_finite_differences(mode):
    inp = small_inputs(T=10, H=8, E=5, k=2, F=4, mode=mode, seed=21 + mode, w_std=0.5)
    # widen the logit gaps so that tiny perturbations cannot change the selection
    inp.w_r = inp.w_r * 4
    dy = O._np(inp.dy)
    fwd = O.layer_forward(inp, rnd=O.identity, exact_logits=True)
    bwd = O.layer_backward(inp, fwd, rnd=O.identity)
    g = np.random.default_rng(1)
    eps = 1e-6
    for name, grad in (("x", bwd["dx"]), ("w_r", bwd["dw_r"]), ("w1", bwd["dw1"]),
                       ("w2", bwd["dw2"])):
        base = getattr(inp, name).to(torch.float64).clone()
        for _ in range(12):
            pos = tuple(int(g.integers(0, s)) for s in base.shape)
            vals = []
            for sgn in (1.0, -1.0):
                pert = base.clone()
                pert[pos] += sgn * eps
                setattr(inp, name, pert)
                L, idx = _loss(inp, dy)
                assert np.array_equal(idx, fwd["idx"])
                vals.append(L)
            setattr(inp, name, base)
            fd = (vals[0] - vals[1]) / (2 * eps)
            assert abs(fd - grad[pos]) <= 1e-6 * max(1.0, abs(fd)), (name, pos, fd, grad[pos])


def test_router_backward_closed_form():
    """dz on the chosen set equals g*(dg - <g,dg>) and is zero elsewhere."""
    inp = small_inputs(T=30, E=7, k=3, seed=4)
    x, w = O._np(inp.x), O._np(inp.w_r)
    z = O.router_logits_fp32(x, w)
    idx, gates = O.route_topk(z, 3)
    dg = np.random.default_rng(0).standard_normal((30, 3))
    dz, _, dw = O.route_bwd(dg, z, idx, x, w, np.zeros_like(x), rnd=O.identity)
    want = np.zeros_like(dz)
    inner = (gates * dg).sum(1, keepdims=True)
    np.put_along_axis(want, idx, gates * (dg - inner), axis=1)
    np.testing.assert_allclose(dz, want, atol=1e-14)
    np.testing.assert_allclose(dw, want.T @ x, atol=1e-12)


def test_backward_chain_fills_every_gradient():
    inp = small_inputs(T=16, H=16, E=4, k=2, F=8, seed=13)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    for key in ("d_o", "dgates", "da", "dx_perm", "dx", "dw_r", "dw1", "dw2"):
        assert np.all(np.isfinite(bwd[key])) and np.abs(bwd[key]).sum() > 0, key


# ----------------------------------------------------------------------------- regression
def test_oracle_regression_fixture():
    """The committed fixture was written by tests/golden/make_oracle_fixture.py (oracle only)."""
    import sys
    sys.path.insert(0, GOLDEN)
    from make_oracle_fixture import compute_fixture
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        stored = json.load(f)
    now = compute_fixture()
    assert now.keys() == stored.keys()
    for key, val in stored.items():
        np.testing.assert_allclose(np.asarray(now[key], np.float64), np.asarray(val, np.float64),
                                   rtol=1e-12, atol=0, err_msg=key)


def test_logit_summation_order_is_ascending_h():
    """The fp32 router sum adds h = 0, 1, 2, ... in turn: 1 + 2^-24 + 2^-24 rounds
    to 1 at each step (ties to even), while the reverse order first makes 2^-23
    and then lands on 1 + 2^-23. Any other order gives a different bit pattern."""
    x = np.array([[1.0, 2.0 ** -24, 2.0 ** -24]])
    w = np.ones((1, 3))
    assert O.router_logits_fp32(x, w)[0, 0] == np.float32(1.0)
    x_rev = x[:, ::-1].copy()
    assert O.router_logits_fp32(x_rev, w)[0, 0] == np.float32(1.0 + 2.0 ** -23)


# ----------------------------------------------------------------------------- wgrad accumulation
def _fd_grad(inp, dy, name, pos, eps=1e-6):
    base = getattr(inp, name).to(torch.float64).clone()
    vals = []
    for sgn in (1.0, -1.0):
        pert = base.clone()
        pert[pos] += sgn * eps
        setattr(inp, name, pert)
        vals.append(_loss(inp, dy)[0])
    setattr(inp, name, base)
    return (vals[0] - vals[1]) / (2 * eps)


def _accum_case(seed=31):
    inp = small_inputs(T=10, H=8, E=5, k=2, F=4, seed=seed, w_std=0.5)
    inp.w_r = inp.w_r * 4
    fwd = O.layer_forward(inp, rnd=O.identity, exact_logits=True)
    bwd = O.layer_backward(inp, fwd, rnd=O.identity)
    rng = np.random.default_rng(seed)
    m1 = rng.standard_normal(tuple(inp.w1.shape)).astype(np.float32)
    m2 = rng.standard_normal(tuple(inp.w2.shape)).astype(np.float32)
    args = (fwd["x_perm"], fwd["h"], bwd["d_o"], bwd["da"], fwd["off"], inp.E)
    return inp, fwd, m1, m2, args


def test_wgrad_accumulation_against_finite_differences():
    """What the accumulation adds to a random fp32 main gradient is the loss's
    gradient, by float64 central differences of the whole layer."""
    inp, fwd, m1, m2, args = _accum_case()
    a1, a2 = O.expert_ffn_bwd_wgrad_accum(m1, m2, *args)
    dy = O._np(inp.dy)
    g = np.random.default_rng(2)
    for name, acc, main in (("w1", a1, m1), ("w2", a2, m2)):
        for _ in range(10):
            pos = tuple(int(g.integers(0, s)) for s in main.shape)
            fd = _fd_grad(inp, dy, name, pos)
            got = float(acc[pos]) - float(main[pos])
            # two fp32 roundings of values of size |main| + |fd|
            tol = 1e-6 * max(1.0, abs(fd)) + 2.4e-7 * (abs(float(main[pos])) + abs(fd))
            assert abs(got - fd) <= tol, (name, pos, got, fd)


def test_wgrad_accumulation_adds_call_after_call():
    """Two calls add the gradient twice, each with one fp32 addition; a zero
    main gradient takes the fp32-rounded gradient exactly."""
    inp, fwd, m1, m2, args = _accum_case(seed=32)
    z1, z2 = O.expert_ffn_bwd_wgrad_accum(np.zeros_like(m1), np.zeros_like(m2), *args)
    b1, b2 = O.expert_ffn_bwd_wgrad_accum(m1, m2, *args)
    c1, c2 = O.expert_ffn_bwd_wgrad_accum(b1, b2, *args)
    for z, m, b, c in ((z1, m1, b1, c1), (z2, m2, b2, c2)):
        assert z.dtype == np.float32 and c.dtype == np.float32
        np.testing.assert_array_equal(b, (m + z).astype(np.float32))
        np.testing.assert_array_equal(c, (b + z).astype(np.float32))
        assert np.abs(z).max() > 0


def test_wgrad_accumulation_leaves_empty_experts_alone():
    inp = small_inputs(T=3, H=8, E=8, k=2, F=4, seed=33)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    cnt = np.diff(fwd["off"])
    assert (cnt == 0).any() and (cnt > 0).any()
    rng = np.random.default_rng(3)
    m1 = rng.standard_normal(tuple(inp.w1.shape)).astype(np.float32)
    m2 = rng.standard_normal(tuple(inp.w2.shape)).astype(np.float32)
    a1, a2 = O.expert_ffn_bwd_wgrad_accum(m1, m2, fwd["x_perm"], fwd["h"], bwd["d_o"],
                                          bwd["da"], fwd["off"], inp.E)
    for e in range(inp.E):
        same = np.array_equal(a1[e], m1[e]) and np.array_equal(a2[e], m2[e])
        assert same == (cnt[e] == 0), e
