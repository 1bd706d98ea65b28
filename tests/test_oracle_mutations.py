"""The pins catch plausible mistakes in the oracle.

Each test plants one mistake in the oracle (on the CPU, by monkeypatching a
function of oracle.moe_oracle for the test's duration) and checks that the pin
meant to guard that step now fails. A pin that still passed with the mistake
in place would not be pinning anything.
"""
import numpy as np
import pytest

import test_oracle_pins as P
from oracle import moe_oracle as O


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


def test_dropped_silu_derivative_term_is_caught(monkeypatch):
    """dgrad with silu'(u) taken as s(u) alone (the u*s*(1-s) term dropped)."""
    def dgrad(d_o, a, off, w1, w2, rnd=O.bf16_rne):
        d_o, a = np.asarray(d_o, np.float64), np.asarray(a, np.float64)
        E, twoF, H = w1.shape
        F = twoF // 2
        da = np.zeros((d_o.shape[0], twoF))
        dx = np.zeros((d_o.shape[0], H))
        for e in range(E):
            r = slice(int(off[e]), int(off[e + 1]))
            dh = d_o[r] @ np.asarray(w2[e], np.float64)
            s = O._sigmoid(a[r, :F])
            da[r, :F] = rnd(dh * a[r, F:] * s)
            da[r, F:] = rnd(dh * a[r, :F] * s)
            dx[r] = rnd(da[r] @ np.asarray(w1[e], np.float64))
        return da, dx
    monkeypatch.setattr(O, "expert_ffn_bwd_dgrad", dgrad)
    _fails(P.test_gradients_against_finite_differences, 0)


def test_swapped_gate_and_up_halves_are_caught(monkeypatch):
    """silu applied to the up half instead of the gate half."""
    orig = O.expert_ffn_fwd

    def fwd(x_perm, off, w1, w2, rnd=O.bf16_rne):
        F = w1.shape[1] // 2
        w1s = np.concatenate([np.asarray(w1)[:, F:], np.asarray(w1)[:, :F]], axis=1)
        return orig(x_perm, off, w1s, w2, rnd)
    monkeypatch.setattr(O, "expert_ffn_fwd", fwd)
    _fails(P.test_single_expert_reduces_to_dense_ffn)


def test_router_gradient_sign_flip_is_caught(monkeypatch):
    orig = O.route_bwd

    def bwd(*a, **kw):
        dz, dx, dw = orig(*a, **kw)
        return -dz, dx, -dw
    monkeypatch.setattr(O, "route_bwd", bwd)
    _fails(P.test_router_backward_closed_form)


def test_unnormalised_gates_are_caught(monkeypatch):
    """Gates left as the softmax probabilities of the chosen experts."""
    monkeypatch.setattr(O, "_renormalised_gates", lambda p, idx: np.take_along_axis(p, idx, axis=1))
    _fails(P.test_gates_equal_softmax_of_selected_logits)
    _fails(P.test_combine_of_dispatch_is_identity)


def test_unstable_layout_is_caught(monkeypatch):
    """Rows of an expert ordered by descending token instead of ascending."""
    orig = O.dispatch_layout

    def layout(idx, E, R=1):
        lay = orig(idx, E, R)
        rs = lay["row_src"].copy()
        for e in range(E):
            seg = slice(int(lay["off"][e]), int(lay["off"][e + 1]))
            rs[seg] = rs[seg][::-1]
        slot = np.empty_like(rs)
        slot[rs] = np.arange(rs.size)
        lay["row_src"], lay["slot"] = rs, slot.reshape(lay["slot"].shape)
        return lay
    monkeypatch.setattr(O, "dispatch_layout", layout)
    _fails(P.test_layout_brute_force_and_invariants, 37, 8, 2, 1, 0)


def test_transposed_wgrad_operand_is_caught(monkeypatch):
    """dW2 built from h rows one step out of line with the d_o rows."""
    orig = O.expert_ffn_bwd_wgrad

    def wgrad(x_perm, h, d_o, da, off, E, rnd=O.bf16_rne):
        return orig(x_perm, np.roll(np.asarray(h, np.float64), 1, axis=0), d_o, da, off, E, rnd)
    monkeypatch.setattr(O, "expert_ffn_bwd_wgrad", wgrad)
    _fails(P.test_gradients_against_finite_differences, 0)


def test_descending_logit_sum_is_caught(monkeypatch):
    orig = O.router_logits_fp32

    def logits(x, w_r, bias=None):
        return orig(np.asarray(x)[:, ::-1], np.asarray(w_r)[:, ::-1], bias)
    monkeypatch.setattr(O, "router_logits_fp32", logits)
    _fails(P.test_logit_summation_order_is_ascending_h)


def test_wgrad_accumulation_that_overwrites_is_caught(monkeypatch):
    """Accumulation that forgets the existing main gradient."""
    orig = O.expert_ffn_bwd_wgrad_accum

    def accum(main_dw1, main_dw2, *args):
        return orig(np.zeros_like(main_dw1), np.zeros_like(main_dw2), *args)
    monkeypatch.setattr(O, "expert_ffn_bwd_wgrad_accum", accum)
    _fails(P.test_wgrad_accumulation_against_finite_differences)
    _fails(P.test_wgrad_accumulation_adds_call_after_call)


def test_wgrad_accumulation_with_a_sign_flip_is_caught(monkeypatch):
    """Accumulation that subtracts the gradient."""
    orig = O.expert_ffn_bwd_wgrad_accum

    def accum(main_dw1, main_dw2, x_perm, h, d_o, da, off, E):
        return orig(main_dw1, main_dw2, x_perm, h, -np.asarray(d_o), -np.asarray(da), off, E)
    monkeypatch.setattr(O, "expert_ffn_bwd_wgrad_accum", accum)
    _fails(P.test_wgrad_accumulation_against_finite_differences)
