"""Seeded synthetic inputs for the MoE layer (x, router/expert weights, dL/dy, router bias).

This module is shared by the CPU oracle and by the CUDA path, so it holds
input synthesis only: it draws numbers and rounds them to the storage dtype.
None of the layer's arithmetic (routing, layout, experts, combine) lives here.

Workloads are the five MoE-layer shapes the EP-overlap pages benchmark
around ("MoE expert-parallel overlap" skill card, benchmark sections: Qwen3
30B-A3B, EP16, BF16, sequence 4096, micro-batch 1, forced-balanced routing),
made synthetic: activations ~N(0,1), weights ~N(0,0.02), rounded to bf16
(round-to-nearest-even, done by torch's dtype conversion).

Layouts (row-major, all "out x in" like a linear layer):
  x   [T, H]      bf16     layer input tokens
  w_r [E, H]      bf16     router weight, logits z = x @ w_r^T (+ bias)
  w1  [E, 2F, H]  bf16     expert FC1; rows 0..F-1 = gate, F..2F-1 = up
  w2  [E, H, F]   bf16     expert FC2
  dy  [T, H]      bf16     upstream gradient dL/dy
  bias [E]        fp32     optional per-expert router bias (skewed routing only)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

ROUTE_SOFTMAX_TOPK = 0
ROUTE_FORCED_BALANCED = 1

SEED_BASE = 20260000

# Named workloads. "id" selects the seed; "mb" > 1 means that many independent
# micro-batches share one set of weights.
WORKLOADS = {
    "tiny": dict(id=1, T=256, H=128, E=8, k=2, F=256, R=1,
                 mode=ROUTE_SOFTMAX_TOPK, bias=None, mb=1),
    "qwen3_30b_a3b_balanced": dict(id=2, T=4096, H=2048, E=128, k=8, F=768, R=1,
                                   mode=ROUTE_FORCED_BALANCED, bias=None, mb=1),
    "qwen3_30b_a3b_skewed": dict(id=3, T=4096, H=2048, E=128, k=8, F=768, R=1,
                                 mode=ROUTE_SOFTMAX_TOPK, bias="zipf_linear", mb=1),
    "ep8_emulated": dict(id=4, T=8192, H=2048, E=64, k=8, F=1408, R=8,
                         mode=ROUTE_SOFTMAX_TOPK, bias=None, mb=1),
    "two_microbatch": dict(id=5, T=4096, H=2048, E=128, k=8, F=768, R=1,
                           mode=ROUTE_FORCED_BALANCED, bias=None, mb=2),
    # parity-only variant of the skewed workload whose bias leaves experts empty
    "qwen3_30b_a3b_skewed_logrank": dict(id=6, T=4096, H=2048, E=128, k=8, F=768, R=1,
                                         mode=ROUTE_SOFTMAX_TOPK, bias="zipf_logrank", mb=1),
}

# independent sub-streams of one workload seed
_S_X, _S_WR, _S_W1, _S_W2, _S_DY, _S_PERM = 0, 1, 2, 3, 4, 5


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def _normal_bf16(seed: int, stream: int, shape, std: float) -> torch.Tensor:
    g = _rng(seed, stream)
    a = g.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).reshape(shape).to(torch.bfloat16)


def zipf_bias(E: int, seed: int, kind: str = "zipf_linear", s: float = 1.1,
              scale: float = 3.0) -> torch.Tensor:
    """Per-expert router bias from a Zipf(s) ranking, mapped onto [-scale, +scale].

    A seeded permutation gives expert e the rank r(e) in 1..E.
    zipf_linear : b_e = -scale + 2*scale*(w(r) - w(E)) / (w(1) - w(E)), w(r) = r^-s
                  (linear in the Zipf weight; the top-ranked expert gets +scale)
    zipf_logrank: b_e = scale - 2*scale*ln(r)/ln(E)
    """
    perm = _rng(seed, _S_PERM).permutation(E)
    rank = np.empty(E, dtype=np.float64)
    rank[perm] = np.arange(1, E + 1, dtype=np.float64)
    if kind == "zipf_linear":
        w = rank ** (-s)
        w1, wE = 1.0, float(E) ** (-s)
        b = -scale + 2.0 * scale * (w - wE) / (w1 - wE) if E > 1 else np.zeros(E)
    elif kind == "zipf_logrank":
        b = scale - 2.0 * scale * np.log(rank) / math.log(E) if E > 1 else np.zeros(E)
    else:
        raise ValueError(f"unknown bias kind {kind!r}")
    return torch.from_numpy(b.astype(np.float32))


@dataclasses.dataclass
class LayerInputs:
    """One micro-batch of synthetic inputs plus the layer's weights (CPU tensors)."""
    T: int
    H: int
    E: int
    k: int
    F: int
    R: int
    mode: int
    x: torch.Tensor
    w_r: torch.Tensor
    w1: torch.Tensor
    w2: torch.Tensor
    dy: torch.Tensor
    bias: Optional[torch.Tensor]
    name: str = ""
    seed: int = 0

    def shape_dict(self):
        return dict(T=self.T, H=self.H, E=self.E, k=self.k, F=self.F, R=self.R, mode=self.mode)


def make_inputs(T: int, H: int, E: int, k: int, F: int, R: int = 1,
                mode: int = ROUTE_SOFTMAX_TOPK, bias: Optional[str] = None,
                seed: int = SEED_BASE, microbatch: int = 0,
                x_std: float = 1.0, w_std: float = 0.02, dy_std: float = 1.0,
                w1_gate_std: Optional[float] = None, name: str = "") -> LayerInputs:
    """Draw one micro-batch's inputs; micro-batch m>0 redraws x and dy only.

    w1_gate_std, when given, is the std of w1's gate rows (rows 0..F-1 of each
    expert) instead of w_std: it widens the gate pre-activations (std about
    w1_gate_std * sqrt(H) for x ~ N(0,1)) to exercise SwiGLU far into both
    tails of the sigmoid. The same normal draws are used, only scaled."""
    xs = _S_X + 16 * microbatch
    ds = _S_DY + 16 * microbatch
    x = _normal_bf16(seed, xs, (T, H), x_std)
    dy = _normal_bf16(seed, ds, (T, H), dy_std)
    w_r = _normal_bf16(seed, _S_WR, (E, H), w_std)
    if w1_gate_std is None:
        w1 = _normal_bf16(seed, _S_W1, (E, 2 * F, H), w_std)
    else:
        g = _rng(seed, _S_W1).standard_normal(E * 2 * F * H, dtype=np.float32)
        g = g.reshape(E, 2 * F, H)
        g[:, :F] *= np.float32(w1_gate_std)
        g[:, F:] *= np.float32(w_std)
        w1 = torch.from_numpy(g).to(torch.bfloat16)
    w2 = _normal_bf16(seed, _S_W2, (E, H, F), w_std)
    b = zipf_bias(E, seed, bias) if bias else None
    return LayerInputs(T=T, H=H, E=E, k=k, F=F, R=R, mode=mode, x=x, w_r=w_r, w1=w1,
                       w2=w2, dy=dy, bias=b, name=name, seed=seed)


def workload(name: str, microbatch: int = 0, T: Optional[int] = None) -> LayerInputs:
    """Inputs of a named workload; T may be lowered to take a token prefix sample."""
    c = WORKLOADS[name]
    inp = make_inputs(T=c["T"], H=c["H"], E=c["E"], k=c["k"], F=c["F"], R=c["R"],
                      mode=c["mode"], bias=c["bias"], seed=SEED_BASE + c["id"],
                      microbatch=microbatch, name=name)
    if T is not None and T < inp.T:
        inp.x = inp.x[:T].contiguous()
        inp.dy = inp.dy[:T].contiguous()
        inp.T = T
    return inp
