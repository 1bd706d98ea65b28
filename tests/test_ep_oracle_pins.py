"""Pins of the EP-exchange oracle (oracle/ep_oracle.py) to facts outside itself:
a hand-worked re-sort, permutation invariants, and the identity that makes an
expert-parallel layer correct: with R ranks exchanging rows, every rank's
outputs and every expert's weight gradient equal those of the single-rank
layer run on all ranks' tokens concatenated in rank order."""
import numpy as np
import pytest
import torch

import moe_synth
from oracle import ep_oracle as EP
from oracle import moe_oracle as O


def test_resort_hand_example():
    # R = 2 sources, E_l = 2 local experts; receive order (source-major):
    #   s0 l0: A | s0 l1: B C | s1 l0: D E | s1 l1: (none)
    recv_cnt = np.array([[1, 2], [2, 0]])
    recv = np.array([[ord(c)] for c in "ABCDE"])
    out, off_local = EP.ep_resort(recv, recv_cnt)
    # expert-major: l0 <- s0 A, s1 D E; l1 <- s0 B C
    assert "".join(chr(v) for v in out[:, 0]) == "ADEBC"
    assert off_local.tolist() == [0, 3, 5]
    assert np.array_equal(EP.ep_unsort(out, recv_cnt), recv)


@pytest.mark.parametrize("R,E_l,seed", [(2, 3, 0), (4, 2, 1), (8, 8, 2), (3, 1, 3)])
def test_resort_is_the_expert_major_permutation(R, E_l, seed):
    g = np.random.default_rng(seed)
    cnt = g.integers(0, 5, size=(R, E_l))
    cnt[g.integers(0, R), :] = 0  # a source that sends nothing
    n = int(cnt.sum())
    # label each row with (source, expert, position) in receive order
    labels = [(s, l, i) for s in range(R) for l in range(E_l) for i in range(cnt[s, l])]
    recv = np.arange(n)[:, None]
    out, off_local = EP.ep_resort(recv, cnt)
    assert sorted(out[:, 0].tolist()) == list(range(n))          # a permutation
    got = [labels[v] for v in out[:, 0]]
    assert got == sorted(labels, key=lambda t: (t[1], t[0], t[2]))  # expert, source, position
    assert np.array_equal(np.diff(off_local), cnt.sum(0))
    assert np.array_equal(EP.ep_unsort(out, cnt), recv)


def test_count_exchange_is_the_transpose_over_ranks():
    g = np.random.default_rng(5)
    R, E_l = 3, 4
    sent = [g.integers(0, 9, size=(R, E_l)) for _ in range(R)]
    got = EP.exchange_counts(sent)
    for d in range(R):
        for s in range(R):
            assert np.array_equal(got[d][s], sent[s][d])


def _ranks(R, T_list, E, k, F, H, seed, mode=0, bias=None):
    base = moe_synth.make_inputs(T=sum(T_list), H=H, E=E, k=k, F=F, R=R, mode=mode, bias=bias,
                                 seed=seed)
    inps, t0 = [], 0
    for T in T_list:
        inp = moe_synth.make_inputs(T=T, H=H, E=E, k=k, F=F, R=R, mode=mode, bias=bias, seed=seed)
        inp.x = base.x[t0:t0 + T].contiguous()
        inp.dy = base.dy[t0:t0 + T].contiguous()
        inps.append(inp)
        t0 += T
    return base, inps


@pytest.mark.parametrize("R,T_list,E,k,mode,bias", [
    (2, [40, 25], 8, 2, 0, None),
    (4, [17, 30, 0, 9], 16, 3, 0, "zipf_logrank"),   # a rank without tokens, empty experts
    # forced balancing routes by token index, (k t + j) mod E, with t counted on
    # each rank; the identity holds when rank 0's k*T is a multiple of E
    (2, [32, 31], 8, 4, 1, None),
])
def test_ep_layer_equals_the_single_rank_layer(R, T_list, E, k, mode, bias):
    H, F = 16, 8
    base, inps = _ranks(R, T_list, E, k, F, H, seed=90 + R, mode=mode, bias=bias)
    ep = EP.ep_layer(inps, R)
    fwd = O.layer_forward(base)
    bwd = O.layer_backward(base, fwd)
    E_l = E // R
    t0 = 0
    for r, T in enumerate(T_list):
        s = ep["src"][r]
        rows = slice(t0, t0 + T)
        # the source's outputs are the single-rank layer's rows of its tokens, bit for bit
        assert np.array_equal(s["y"], fwd["y"][rows])
        assert np.array_equal(s["dx"], bwd["dx"][rows])
        assert np.array_equal(s["idx"], fwd["idx"][rows])
        t0 += T
    # every owner's expert-major rows are the single-rank layout's rows of its experts
    for d in range(R):
        w = ep["own"][d]
        lo, hi = int(fwd["off"][d * E_l]), int(fwd["off"][(d + 1) * E_l])
        assert np.array_equal(w["x_sorted"], fwd["x_perm"][lo:hi])
        assert np.array_equal(w["off_local"], fwd["off"][d * E_l:(d + 1) * E_l + 1] - lo)
        # the expert weight gradients, each reduced over every rank's rows
        assert np.array_equal(w["dw1"], bwd["dw1"][d * E_l:(d + 1) * E_l])
        assert np.array_equal(w["dw2"], bwd["dw2"][d * E_l:(d + 1) * E_l])
    # the router weight gradient is the sum of the sources' (float64, order differs)
    dwr = sum(s["dw_r"] for s in ep["src"])
    np.testing.assert_allclose(dwr, bwd["dw_r"], rtol=1e-12, atol=1e-14)
    # every routed row goes out and comes back once: row counts balance
    sent = sum(int(s["rank_off"][-1]) for s in ep["src"])
    recv = sum(int(w["off_local"][-1]) for w in ep["own"])
    assert sent == recv == sum(T_list) * k


def test_ep_layer_with_one_rank_is_the_layer():
    base, inps = _ranks(1, [37], 6, 2, 8, 16, seed=95)
    ep = EP.ep_layer(inps, 1)
    fwd = O.layer_forward(base)
    assert np.array_equal(ep["x_recv"][0], fwd["x_perm"])
    assert np.array_equal(ep["src"][0]["y"], fwd["y"])
