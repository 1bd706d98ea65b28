"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle on the same seeded inputs.

Tolerance (floats): per tensor, max |gpu - oracle| / max |oracle| <= 2e-2 for
bf16 inputs with fp32 accumulation (the layer's stated bar). Integers
(routing indices, counts, offsets, slots, the inverse permutation and the
per-rank tables) must match exactly.

Element-wise error: max_i |gpu_i - oracle_i| / max(|oracle_i|, 1e-3 * rms(oracle)).
It is reported for every float tensor of a whole-layer run, where it also
carries the conditioning of the chain: a one-ulp difference of a bf16 gate
pre-activation a_g moves silu(a_g) by |1 + a_g (1 - s(a_g))| ulps (nine at
a_g = -10), and one rounding flip of a large da moves the small elements of
dx_perm by ~1e-3 of its rms. Element by element the layer is therefore
checked stage by stage (check_stages): each expert stage is re-run by the
oracle on the GPU's own stored inputs of that stage, so the only differences
left are the stage's fp32 arithmetic and one bf16 rounding on each side.
"""
from __future__ import annotations

import numpy as np
import torch

import combine_router_softmax_top_gb300 as moe
from oracle import moe_oracle as O

TOL = 2e-2


def desc_of(inp) -> moe.LayerDesc:
    return moe.LayerDesc.of(T=inp.T, H=inp.H, E=inp.E, k=inp.k, F=inp.F, R=inp.R, mode=inp.mode)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def npi(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def rel_err(gpu, ora) -> float:
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    if ora.size == 0:
        return 0.0
    scale = max(float(np.abs(ora).max()), 1e-6)
    return float(np.abs(gpu - ora).max()) / scale


def elem_rel_err(gpu, ora, floor=1e-3) -> float:
    """max_i |gpu_i - ora_i| / max(|ora_i|, floor * rms(ora))."""
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    if ora.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ora * ora)))
    den = np.maximum(np.abs(ora), max(floor * rms, 1e-30))
    return float((np.abs(gpu - ora) / den).max())


def assert_close(name, gpu, ora, tol=TOL):
    err = rel_err(gpu, ora)
    assert np.all(np.isfinite(np.asarray(gpu, np.float64))), f"{name}: non-finite values"
    assert err <= tol, f"{name}: max relative error {err:.3e} > {tol}"
    return err


def assert_equal(name, gpu, ora):
    gpu = np.asarray(gpu)
    ora = np.asarray(ora)
    assert gpu.shape == ora.shape, f"{name}: shape {gpu.shape} vs {ora.shape}"
    bad = np.flatnonzero(gpu.reshape(-1) != ora.reshape(-1))
    assert bad.size == 0, f"{name}: {bad.size} mismatches, first at {bad[:5]}"


def run_layer(inp, device="cuda", run_wgrad=True) -> dict:
    """Forward + backward through moe_layer_forward / moe_layer_backward."""
    d = desc_of(inp)
    b = moe.LayerBuffers(d, device)
    b.load_inputs(inp)
    moe.moe_layer_forward(d, b)
    moe.moe_layer_backward(d, b, run_wgrad=run_wgrad)
    st = moe.moe_device_status(d, b.ws)
    assert st == moe.MOE_OK, moe.lib().moe_last_error()
    torch.cuda.synchronize()
    return collect(b, inp)


def collect(b, inp) -> dict:
    T, k = inp.T, inp.k
    N = T * k
    out = {}
    for name in ("idx", "slot"):
        out[name] = npi(getattr(b, name))[:T]
    out["row_src"] = npi(b.row_src)[:N]
    for name in ("cnt", "off", "cnt_re", "rank_off"):
        out[name] = npi(getattr(b, name))
    out["logits"] = b.logits.detach().cpu().numpy()[:T]
    for name in ("gates", "dgates"):
        out[name] = np64(getattr(b, name))[:T]
    for name in ("x_perm", "a", "h", "o", "d_o", "da", "dx_perm"):
        out[name] = np64(getattr(b, name))[:N]
    for name in ("y", "dx", "dx32"):
        out[name] = np64(getattr(b, name))[:T]
    for name in ("dw_r", "dw1", "dw2", "main_dw1", "main_dw2"):
        t = getattr(b, name)
        if t is not None:
            out[name] = np64(t)
    return out


def oracle_layer(inp) -> dict:
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    return {**fwd, **bwd}


INT_KEYS = ("idx", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off")
FLOAT_KEYS = ("gates", "x_perm", "a", "h", "o", "y", "d_o", "dgates", "da", "dx_perm", "dx",
              "dw_r", "dw1", "dw2")


def compare_layer(g: dict, o: dict, skip=(), elementwise: dict = None) -> dict:
    """Exact integer parity, tolerance float parity; returns the float errors.
    When a dict is passed as `elementwise`, it receives the element-wise errors."""
    for key in INT_KEYS:
        if key not in skip:
            assert_equal(key, g[key], o[key])
    # the router logits are the fixed-order fp32 sums on both sides
    if "logits" not in skip:
        assert_equal("logits", g["logits"].view(np.uint32), np.asarray(o["z"], np.float32).view(np.uint32))
    errs = {}
    for key in FLOAT_KEYS:
        if key not in skip:
            ref = o["dx_experts"] if key == "dx32" else o[key]
            errs[key] = assert_close(key, g[key], ref)
            if elementwise is not None:
                elementwise[key] = elem_rel_err(g[key], ref)
    return errs


U32 = 2.0 ** -24  # fp32 unit roundoff


def _within_bound(got, ref, acc) -> float:
    """max_i |got_i - ref_i| / tol_i with tol_i = 2^-7 (1 + 2^-7) |ref_i| + acc_i:
    one bf16 ulp between two roundings of nearby values, plus acc_i, the fp32
    error of the value before its rounding. <= 1 passes."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    tol = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(ref) + acc
    err = np.abs(got - ref)
    ratio = np.where(err == 0, 0.0, err / np.maximum(tol, 1e-300))
    return float(ratio.max())


def check_stages(g: dict, inp, tol=TOL) -> dict:
    """Element by element, each expert stage against the oracle's stage function
    re-run on the GPU's own stored inputs of that stage:
      a        = expert_fc1_fwd(x_perm)            from the GPU's x_perm
      h        = swiglu(a)                         from the GPU's a
      o        = expert_fc2_fwd(h)                 from the GPU's h
      da       = expert_fc2_dgrad(d_o, a)          from the GPU's d_o and a
      dx_perm  = expert_fc1_dgrad(da)              from the GPU's da
    Both sides round the same value to bf16, so each element may differ by one
    bf16 ulp (2^-7 of the value at most) plus the GPU's fp32 error before the
    rounding. For a K-term product that error is taken as 4 sqrt(K) 2^-24
    sum_k |a_k b_k| (four times the root-K scale of fp32 accumulation error;
    sum_k |a_k b_k| is the same stage function run on absolute values), carried
    through the SwiGLU gradient's factor for da; the elementwise SwiGLU itself
    adds 2^-20 of the value (a few fp32 roundings and the fast exp/divide).
    Asserts every element within that bound. Returns, per stage, the bound
    ratio (<= 1) and the element-wise relative error with the 1e-3 rms floor."""
    w1, w2 = O._np(inp.w1), O._np(inp.w2)
    aw1, aw2 = np.abs(w1), np.abs(w2)
    off = np.asarray(g["off"], np.int64)
    N = int(off[-1])
    st = {k: g[k][:N] for k in ("x_perm", "a", "h", "o", "d_o", "da", "dx_perm")}
    H, F = inp.H, inp.F
    ident = O.identity
    ref = {
        "a": O.expert_fc1_fwd(st["x_perm"], off, w1),
        "h": O.swiglu(st["a"]),
        "o": O.expert_fc2_fwd(st["h"], off, w2),
        "da": O.expert_fc2_dgrad(st["d_o"], st["a"], off, w2),
        "dx_perm": O.expert_fc1_dgrad(st["da"], off, w1),
    }
    elem = 2.0 ** -20
    acc = {
        "a": 4 * np.sqrt(H) * U32 * O.expert_fc1_fwd(np.abs(st["x_perm"]), off, aw1, ident),
        "h": elem * np.abs(O.swiglu(st["a"], ident)),
        "o": 4 * np.sqrt(F) * U32 * O.expert_fc2_fwd(np.abs(st["h"]), off, aw2, ident),
        "da": 4 * np.sqrt(H) * U32 * np.abs(O.expert_fc2_dgrad(np.abs(st["d_o"]), st["a"], off,
                                                                aw2, ident))
              + elem * np.abs(O.expert_fc2_dgrad(st["d_o"], st["a"], off, w2, ident)),
        "dx_perm": 4 * np.sqrt(2 * F) * U32 * O.expert_fc1_dgrad(np.abs(st["da"]), off, aw1, ident),
    }
    out = {}
    for key in ref:
        ratio = _within_bound(st[key], ref[key], acc[key])
        out[key] = {"bound_ratio": ratio, "elem": elem_rel_err(st[key], ref[key])}
        assert ratio <= 1.0, (f"{key}: an element differs from the oracle's stage by "
                              f"{ratio:.2f} x (one bf16 ulp + fp32 error)")
    return out
