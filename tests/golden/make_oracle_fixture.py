"""Writes oracle_small.json: a regression record of the oracle on one small case.

It calls only the oracle (and the seeded input generator), so a later change to
the oracle's arithmetic shows up as a fixture mismatch and must be justified.
Run from the repository root:  python tests/golden/make_oracle_fixture.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_synth  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402


def compute_fixture():
    inp = moe_synth.make_inputs(T=12, H=64, E=4, k=2, F=64, R=2, seed=424242)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    out = {"idx": fwd["idx"].tolist(), "slot": fwd["slot"].tolist(),
           "gates": fwd["gates"].tolist(), "y_row0": fwd["y"][0].tolist(),
           "dx_row0": bwd["dx"][0].tolist(), "dgates": bwd["dgates"].tolist()}
    for key in ("a", "h", "o", "y", "d_o", "da", "dx_perm", "dx"):
        arr = fwd[key] if key in fwd else bwd[key]
        out[key + "_sum"] = float(arr.sum())
        out[key + "_sumsq"] = float((arr * arr).sum())
    for key in ("dw_r", "dw1", "dw2"):
        out[key + "_sum"] = float(bwd[key].sum())
        out[key + "_sumsq"] = float((bwd[key] ** 2).sum())
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(compute_fixture(), f, indent=1)
