"""CPU oracle of one MoE layer: route, dispatch layout, permute, expert SwiGLU FFN,
combine, and the backward split into dgrad and wgrad.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module; only
the tests, the package's smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA path: the one module both sides use is
``moe_synth`` (seeded input synthesis, no layer arithmetic).

What the pages fix, and what they leave open
--------------------------------------------
The EP-overlap pages ("MoE expert-parallel overlap" skill card; the obnotes
"1. MoE EP Overlap" note) give the layer's structure, not its arithmetic:
  * the MoE part of a layer runs as the phases dispatch -> mlp -> combine
    (obnotes, section "how the 8 fwd/bwd operations are split out");
  * backward runs combine -> mlp -> dispatch (same section, the manual backward
    chain), with the mlp backward split so the activation gradient (dgrad) is
    produced first and the weight gradient (wgrad) can be deferred
    (obnotes, section "MoE 1F1B overlap"; skill card, section "what it is",
    delay_wgrad_compute);
  * the dispatcher is the standard MoE all-to-all (skill card, "what it is",
    dispatcher table), benchmarked with BF16 and force-balanced routing
    (skill card, "HybridEP production benchmark").
The arithmetic follows the layer definition this library implements:
router logits in fp32, softmax over all experts, top-k, gates renormalised over
the chosen k, dropless dispatch, SwiGLU experts, gate-weighted combine.
Readings taken where that definition is silent (each also listed in the design
notes):
  R1 logits: z[t,e] = sum over h = 0..H-1 in ascending order, fp32, starting from
     0; bf16*bf16 products are exact in fp32, so each step is one fp32 rounding.
     A per-expert bias, when present, is added afterwards in fp32.
  R2 top-k is taken on the fp32 logits (softmax is monotone), descending, ties to
     the lower expert index; slot j = 0..k-1 follows that order.
  R3 gates: p = softmax over all E experts; g_j = p[i_j] / sum_l p[i_l].
  R4 forced balancing: i_j = (k*t + j) mod E, gates from the same p renormalised
     over that set.
  R5 layout: rows of one expert are contiguous, experts ascending, and within an
     expert rows ascend by token (stable); no padding. With R emulated ranks,
     rank(e) = e div (E/R), so rank-major expert-contiguous order is expert order.
  R6 SwiGLU: h = silu(a_gate) * a_up, W1 rows 0..F-1 gate, F..2F-1 up; no biases.
  R7 combine and unpermute sum over j = 0..k-1; the layer's input gradient is the
     expert path's plus the router's: dx = bf16(sum_j dx_perm + dz @ w_r).
  R8 stored tensors are bf16 (round to nearest even) at: a, h, o, y, d_o, da,
     dx_perm, dx, dW1, dW2. Gates, dgates, dz and dW_r are kept in high precision.
  R13 gradient accumulation fusion (optional): the expert weight gradients, rounded
      once to fp32, are added into fp32 main gradients with one fp32 addition per
      element, call after call; an expert with no rows adds nothing.
Everything else is computed in float64; ``rnd=identity`` turns the bf16 rounding
off for the finite-difference pins.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_rne", "identity", "router_logits_fp32", "router_logits_exact", "route_topk",
    "route_forced", "softmax_full", "dispatch_layout", "permute", "swiglu", "swiglu_bwd",
    "expert_fc1_fwd", "expert_fc2_fwd", "expert_ffn_fwd", "expert_fc2_dgrad", "expert_fc1_dgrad",
    "combine", "combine_bwd", "expert_ffn_bwd_dgrad", "expert_ffn_bwd_wgrad",
    "expert_ffn_bwd_wgrad_accum", "permute_bwd", "route_bwd", "layer_forward", "layer_backward",
]


# ----------------------------------------------------------------------------- rounding
def bf16_rne(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even (R8).

    Works on the float64 bit pattern directly (no intermediate fp32 rounding):
    bf16 keeps 7 explicit mantissa bits, float64 has 52, so the low 45 bits are
    rounded off. Exponent range and NaN/inf are left as float64 has them; the
    layer's values never approach the fp32 exponent limits.
    """
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = a.view(np.uint64).copy()
    finite = np.isfinite(a)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = b + (np.uint64((1 << 44) - 1) + lsb)
    b &= ~np.uint64((1 << 45) - 1)
    out = b.view(np.float64)
    return np.where(finite, out, a)


def identity(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _silu(u):
    return u / (1.0 + np.exp(-u))


def _sigmoid(u):
    return 1.0 / (1.0 + np.exp(-u))


def swiglu(a, rnd=bf16_rne) -> np.ndarray:
    """h = rnd(silu(a_gate) * a_up) for rows a = [a_gate | a_up] of width 2F (R6)."""
    a = np.asarray(a, np.float64)
    F = a.shape[1] // 2
    return rnd(_silu(a[:, :F]) * a[:, F:])


def swiglu_bwd(dh, a, rnd=bf16_rne) -> np.ndarray:
    """Gradient of swiglu at a for the upstream dh [rows, F]:
    da_gate = rnd(dh * a_up * silu'(a_gate)), silu'(u) = s(u) * (1 + u * (1 - s(u)));
    da_up = rnd(dh * silu(a_gate)), with s the logistic sigmoid."""
    dh = np.asarray(dh, np.float64)
    a = np.asarray(a, np.float64)
    F = a.shape[1] // 2
    ag, au = a[:, :F], a[:, F:]
    s = _sigmoid(ag)
    da = np.empty_like(a)
    da[:, :F] = rnd(dh * au * s * (1.0 + ag * (1.0 - s)))
    da[:, F:] = rnd(dh * ag * s)
    return da


# ----------------------------------------------------------------------------- route
def router_logits_fp32(x, w_r, bias=None) -> np.ndarray:
    """Router logits in fp32 with the fixed summation order of R1.

    x [T,H], w_r [E,H] hold bf16 values. Returns z [T,E] float32.
    """
    x32 = np.asarray(x, dtype=np.float32)
    w32 = np.asarray(w_r, dtype=np.float32)
    T, H = x32.shape
    E = w32.shape[0]
    z = np.zeros((T, E), dtype=np.float32)
    for h in range(H):  # ascending h, one fp32 add per step; x*w is exact in fp32
        z += np.outer(x32[:, h], w32[:, h])
    if bias is not None:
        z += np.asarray(bias, dtype=np.float32)[None, :]
    return z


def router_logits_exact(x, w_r, bias=None) -> np.ndarray:
    """Router logits in float64 (used only by the finite-difference pins)."""
    z = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T
    if bias is not None:
        z = z + np.asarray(bias, np.float64)[None, :]
    return z


def softmax_full(z) -> np.ndarray:
    """p = softmax over all experts, per token (R3), in float64."""
    z = np.asarray(z, np.float64)
    m = z.max(axis=1, keepdims=True)
    ez = np.exp(z - m)
    return ez / ez.sum(axis=1, keepdims=True)


def _renormalised_gates(p, idx):
    sel = np.take_along_axis(p, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route_topk(z, k: int):
    """Top-k experts per token by logit (R2) and renormalised gates (R3)."""
    z = np.asarray(z)
    # a stable sort of -z keeps ascending expert order among equal logits
    idx = np.argsort(-z, axis=1, kind="stable")[:, :k].astype(np.int32)
    gates = _renormalised_gates(softmax_full(z), idx)
    return idx, gates


def route_forced(z, k: int):
    """Force-balanced routing (R4): token t goes to experts (k*t + j) mod E."""
    z = np.asarray(z)
    T, E = z.shape
    t = np.arange(T, dtype=np.int64)[:, None]
    j = np.arange(k, dtype=np.int64)[None, :]
    idx = ((k * t + j) % E).astype(np.int32)
    gates = _renormalised_gates(softmax_full(z), idx)
    return idx, gates


# ----------------------------------------------------------------------------- dispatch
def dispatch_layout(idx, E: int, R: int = 1):
    """Dropless dispatch layout (R5).

    Returns dict with
      cnt [E]       rows per expert
      off [E+1]     exclusive prefix of cnt (expert e owns rows off[e]..off[e+1]-1)
      slot [T,k]    row of (t, j) in the permuted buffer
      row_src [N]   inverse of slot: row_src[slot[t,j]] = t*k + j
      cnt_re [R,E/R] rows per (rank, local expert): the counts an EP all-to-all exchanges
      rank_off [R+1] first row of each rank's chunk of the send buffer
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    N = T * k
    flat = idx.reshape(-1).astype(np.int64)
    cnt = np.bincount(flat, minlength=E).astype(np.int64)
    off = np.zeros(E + 1, dtype=np.int64)
    off[1:] = np.cumsum(cnt)
    # entries ordered by expert; the stable sort keeps ascending t*k+j inside an expert
    row_src = np.argsort(flat, kind="stable").astype(np.int64)
    slot = np.empty(N, dtype=np.int64)
    slot[row_src] = np.arange(N, dtype=np.int64)
    E_l = E // R
    cnt_re = cnt.reshape(R, E_l)
    rank_off = off[np.arange(R + 1) * E_l]
    return dict(cnt=cnt, off=off, slot=slot.reshape(T, k), row_src=row_src,
                cnt_re=cnt_re, rank_off=rank_off)


def permute(x, row_src, k: int) -> np.ndarray:
    """EP send buffer: x_perm[s] = x[row_src[s] div k] (dispatch phase)."""
    x = np.asarray(x, np.float64)
    return x[np.asarray(row_src) // k]


# ----------------------------------------------------------------------------- experts
def _per_expert(off, rows_out, fn):
    """Runs fn(e, r) for every expert e with rows r = off[e]..off[e+1]-1."""
    for e in range(len(off) - 1):
        r = slice(int(off[e]), int(off[e + 1]))
        if r.stop > r.start:
            rows_out[r] = fn(e, r)
    return rows_out


def expert_fc1_fwd(x_perm, off, w1, rnd=bf16_rne):
    """a = rnd(x_e @ W1_e^T) per expert (the first GEMM of the mlp phase, R6)."""
    x_perm = np.asarray(x_perm, np.float64)
    a = np.zeros((x_perm.shape[0], w1.shape[1]))
    return _per_expert(off, a, lambda e, r: rnd(x_perm[r] @ np.asarray(w1[e], np.float64).T))


def expert_fc2_fwd(h, off, w2, rnd=bf16_rne):
    """o = rnd(h_e @ W2_e^T) per expert (the second GEMM of the mlp phase)."""
    h = np.asarray(h, np.float64)
    o = np.zeros((h.shape[0], w2.shape[1]))
    return _per_expert(off, o, lambda e, r: rnd(h[r] @ np.asarray(w2[e], np.float64).T))


def expert_ffn_fwd(x_perm, off, w1, w2, rnd=bf16_rne):
    """Per-expert SwiGLU FFN on the expert-contiguous rows (mlp phase, R6).

    a = rnd(x_e @ W1_e^T); h = rnd(silu(a_gate) * a_up); o = rnd(h @ W2_e^T).
    Rows outside every expert's range (none in a dropless layout) stay 0.
    """
    a = expert_fc1_fwd(x_perm, off, w1, rnd)
    h = np.zeros((a.shape[0], a.shape[1] // 2))
    _per_expert(off, h, lambda e, r: swiglu(a[r], rnd))
    o = expert_fc2_fwd(h, off, w2, rnd)
    return a, h, o


def combine(o, slot, gates, rnd=bf16_rne) -> np.ndarray:
    """y[t] = rnd(sum_j g[t,j] * o[slot[t,j]]), j ascending (combine phase, R7)."""
    o = np.asarray(o, np.float64)
    slot = np.asarray(slot)
    gates = np.asarray(gates, np.float64)
    T, k = slot.shape
    y = np.zeros((T, o.shape[1]))
    for j in range(k):
        y += gates[:, j:j + 1] * o[slot[:, j]]
    return rnd(y)


def combine_bwd(dy, o, slot, gates, rnd=bf16_rne):
    """Backward of combine: d_o[slot[t,j]] = rnd(g[t,j]*dy[t]); dg[t,j] = <dy[t], o[slot[t,j]]>."""
    dy = np.asarray(dy, np.float64)
    o = np.asarray(o, np.float64)
    slot = np.asarray(slot)
    gates = np.asarray(gates, np.float64)
    T, k = slot.shape
    d_o = np.zeros_like(o)
    dgates = np.zeros((T, k))
    for j in range(k):
        d_o[slot[:, j]] = rnd(gates[:, j:j + 1] * dy)
        dgates[:, j] = np.einsum("th,th->t", dy, o[slot[:, j]])
    return d_o, dgates


def expert_fc2_dgrad(d_o, a, off, w2, rnd=bf16_rne):
    """da = swiglu_bwd(d_o_e @ W2_e, a_e) per expert: the gradient through the
    second GEMM and the SwiGLU (dh is not rounded; da is)."""
    d_o = np.asarray(d_o, np.float64)
    a = np.asarray(a, np.float64)
    da = np.zeros_like(a)
    return _per_expert(off, da, lambda e, r: swiglu_bwd(d_o[r] @ np.asarray(w2[e], np.float64),
                                                        a[r], rnd))


def expert_fc1_dgrad(da, off, w1, rnd=bf16_rne):
    """dx_perm = rnd(da_e @ W1_e) per expert: the gradient through the first GEMM."""
    da = np.asarray(da, np.float64)
    dx = np.zeros((da.shape[0], w1.shape[2]))
    return _per_expert(off, dx, lambda e, r: rnd(da[r] @ np.asarray(w1[e], np.float64)))


def expert_ffn_bwd_dgrad(d_o, a, off, w1, w2, rnd=bf16_rne):
    """Activation gradient of the experts (the part computed before wgrad).

    dh = d_o_e @ W2_e; da_up = dh * silu(a_g); da_gate = dh * a_u * silu'(a_g),
    silu'(u) = s(u) * (1 + u * (1 - s(u))); dx_perm = rnd(rnd(da) @ W1_e).
    """
    da = expert_fc2_dgrad(d_o, a, off, w2, rnd)
    return da, expert_fc1_dgrad(da, off, w1, rnd)


def expert_ffn_bwd_wgrad(x_perm, h, d_o, da, off, E: int, rnd=bf16_rne):
    """Weight gradients of the experts (the deferrable part).

    dW1_e = rnd(da_e^T @ x_e), dW2_e = rnd(d_o_e^T @ h_e); an expert with no rows
    gets zeros.
    """
    x_perm = np.asarray(x_perm, np.float64)
    h = np.asarray(h, np.float64)
    d_o = np.asarray(d_o, np.float64)
    da = np.asarray(da, np.float64)
    twoF, H, F = da.shape[1], x_perm.shape[1], h.shape[1]
    dw1 = np.zeros((E, twoF, H))
    dw2 = np.zeros((E, H, F))
    for e in range(E):
        r = slice(int(off[e]), int(off[e + 1]))
        if r.stop == r.start:
            continue
        dw1[e] = rnd(da[r].T @ x_perm[r])
        dw2[e] = rnd(d_o[r].T @ h[r])
    return dw1, dw2


def expert_ffn_bwd_wgrad_accum(main_dw1, main_dw2, x_perm, h, d_o, da, off, E: int):
    """Weight gradients added into fp32 main gradients (gradient accumulation fusion).

    The skill card lists gradient_accumulation_fusion beside delay_wgrad_compute
    (section "compatibility and constraints", and the troubleshooting table),
    and the "1. MoE EP Overlap" note runs the backward with accumulate_grad=True,
    which adds into the existing gradient instead of overwriting it. Reading:
    the expert's weight gradient, computed exactly (float64) and rounded once to
    fp32, is added to the fp32 main gradient with one fp32 addition:
      main_dw1[e] <- fp32(main_dw1[e] + fp32(da_e^T @ x_e))
      main_dw2[e] <- fp32(main_dw2[e] + fp32(d_o_e^T @ h_e))
    An expert with no rows adds nothing. Returns new float32 arrays.
    """
    m1 = np.array(main_dw1, dtype=np.float32, copy=True)
    m2 = np.array(main_dw2, dtype=np.float32, copy=True)
    x_perm = np.asarray(x_perm, np.float64)
    h = np.asarray(h, np.float64)
    d_o = np.asarray(d_o, np.float64)
    da = np.asarray(da, np.float64)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        g1 = (da[lo:hi].T @ x_perm[lo:hi]).astype(np.float32)
        g2 = (d_o[lo:hi].T @ h[lo:hi]).astype(np.float32)
        m1[e] = m1[e] + g1  # float32 + float32: one fp32 rounding
        m2[e] = m2[e] + g2
    return m1, m2


def permute_bwd(dx_perm, slot) -> np.ndarray:
    """Backward of dispatch: dx_e[t] = sum_j dx_perm[slot[t,j]] (not rounded)."""
    dx_perm = np.asarray(dx_perm, np.float64)
    slot = np.asarray(slot)
    T, k = slot.shape
    dx = np.zeros((T, dx_perm.shape[1]))
    for j in range(k):
        dx += dx_perm[slot[:, j]]
    return dx


def route_bwd(dgates, z, idx, x, w_r, dx_experts, rnd=bf16_rne):
    """Backward of the router through the renormalised gates.

    The gates are g = P[idx] / sum(P[idx]) with P = softmax(z) over all E. The
    chain rule is written out over the full softmax: dP/dz = diag(P) - P P^T and
    dg_j/dP_i = ([i = i_j] - g_j [i in S]) / sum_S P.  Then
      dz = (dg/dz)^T dgates,  dx = rnd(dx_experts + dz @ w_r),  dW_r = dz^T @ x.
    Returns dz [T,E], dx [T,H], dw_r [E,H].
    """
    dgates = np.asarray(dgates, np.float64)
    x = np.asarray(x, np.float64)
    w_r = np.asarray(w_r, np.float64)
    idx = np.asarray(idx)
    P = softmax_full(z)
    T, E = P.shape
    k = idx.shape[1]
    dz = np.zeros((T, E))
    for t in range(T):
        S = idx[t]
        pS = P[t, S]
        sumS = pS.sum()
        g = pS / sumS
        dg_dP = np.zeros((k, E))
        for j in range(k):
            dg_dP[j, S] -= g[j] / sumS
            dg_dP[j, S[j]] += 1.0 / sumS
        dP_dz = np.diag(P[t]) - np.outer(P[t], P[t])
        dz[t] = (dg_dP @ dP_dz).T @ dgates[t]
    dx = rnd(np.asarray(dx_experts, np.float64) + dz @ w_r)
    dw_r = dz.T @ x
    return dz, dx, dw_r


# ----------------------------------------------------------------------------- layer
def _np(t):
    """torch tensor / array -> float64 numpy (bf16 values are exact in float64)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def layer_forward(inp, rnd=bf16_rne, exact_logits: bool = False):
    """Forward of one MoE layer on ``moe_synth.LayerInputs``-like inputs.

    Phases in page order: route (router), dispatch (layout + permute), mlp
    (expert FFN), combine. Returns a dict with every saved tensor.
    """
    x, w_r, w1, w2 = _np(inp.x), _np(inp.w_r), _np(inp.w1), _np(inp.w2)
    bias = None if inp.bias is None else _np(inp.bias)
    if exact_logits:
        z = router_logits_exact(x, w_r, bias)
    else:
        z = router_logits_fp32(x, w_r, bias)
    if inp.mode == 1:
        idx, gates = route_forced(z, inp.k)
    else:
        idx, gates = route_topk(z, inp.k)
    lay = dispatch_layout(idx, inp.E, inp.R)
    x_perm = permute(x, lay["row_src"], inp.k)
    a, h, o = expert_ffn_fwd(x_perm, lay["off"], w1, w2, rnd)
    y = combine(o, lay["slot"], gates, rnd)
    return dict(z=z, idx=idx, gates=gates, x_perm=x_perm, a=a, h=h, o=o, y=y, **lay)


def layer_backward(inp, fwd, rnd=bf16_rne, dy=None):
    """Backward in the pages' chain order: combine -> mlp (dgrad) -> dispatch -> router,
    then the deferred expert wgrad."""
    x, w_r, w1, w2 = _np(inp.x), _np(inp.w_r), _np(inp.w1), _np(inp.w2)
    dy = _np(inp.dy) if dy is None else np.asarray(dy, np.float64)
    d_o, dgates = combine_bwd(dy, fwd["o"], fwd["slot"], fwd["gates"], rnd)
    da, dx_perm = expert_ffn_bwd_dgrad(d_o, fwd["a"], fwd["off"], w1, w2, rnd)
    dx_e = permute_bwd(dx_perm, fwd["slot"])
    dz, dx, dw_r = route_bwd(dgates, fwd["z"], fwd["idx"], x, w_r, dx_e, rnd)
    dw1, dw2 = expert_ffn_bwd_wgrad(fwd["x_perm"], fwd["h"], d_o, da, fwd["off"], inp.E, rnd)
    return dict(d_o=d_o, dgates=dgates, da=da, dx_perm=dx_perm, dx_experts=dx_e, dz=dz,
                dx=dx, dw_r=dw_r, dw1=dw1, dw2=dw2)
