"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle on the same seeded inputs.

Tolerance (floats): per tensor, max |gpu - oracle| / max |oracle| <= 2e-2 for
bf16 inputs with fp32 accumulation (the layer's stated bar). Integers
(routing indices, counts, offsets, slots, the inverse permutation and the
per-rank tables) must match exactly.
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
    for name in ("dw_r", "dw1", "dw2"):
        out[name] = np64(getattr(b, name))
    return out


def oracle_layer(inp) -> dict:
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    return {**fwd, **bwd}


INT_KEYS = ("idx", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off")
FLOAT_KEYS = ("gates", "x_perm", "a", "h", "o", "y", "d_o", "dgates", "da", "dx_perm", "dx",
              "dw_r", "dw1", "dw2")


def compare_layer(g: dict, o: dict, skip=()) -> dict:
    """Exact integer parity, tolerance float parity; returns the float errors."""
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
    return errs
