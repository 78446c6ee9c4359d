"""Writes tiny_causal_gqa.txt: dQ, dK, dV of a tiny causal GQA case evaluated by
the oracle alone (float64 forward and backward), as a regression fixture for the
oracle.  Inputs come from the seeded generator; nothing here touches the CUDA
library.  Run from the repository root:  python tests/golden/make_tiny.py"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_backward_gb300 import inputs  # noqa: E402

CASE = dict(B=1, S=6, HQ=4, HKV=2, D=3, seed=777, scale=0.5, window=4)


def tiny_inputs():
    c = CASE
    q = inputs.normal_f32(c["seed"], 0, (c["B"], c["S"], c["HQ"], c["D"])).astype(np.float64)
    k = inputs.normal_f32(c["seed"], 1, (c["B"], c["S"], c["HKV"], c["D"])).astype(np.float64)
    v = inputs.normal_f32(c["seed"], 2, (c["B"], c["S"], c["HKV"], c["D"])).astype(np.float64)
    do = inputs.normal_f32(c["seed"], 3, (c["B"], c["S"], c["HQ"], c["D"])).astype(np.float64)
    return q, k, v, do


def evaluate():
    q, k, v, do = tiny_inputs()
    mask = dict(causal=True, window=CASE["window"])
    o, lse = oracle.forward(q, k, v, CASE["scale"], dtype=np.float64, **mask)
    return oracle.backward(q, k, v, o, do, lse, CASE["scale"], **mask)


def main():
    dq, dk, dv = evaluate()
    lines = ["# dQ, dK, dV of the case below, evaluated by the oracle in float64 (make_tiny.py).",
             "# " + " ".join(f"{a}={b}" for a, b in CASE.items())]
    for name, arr in (("dq", dq), ("dk", dk), ("dv", dv)):
        lines.append(f"{name} {' '.join(str(x) for x in arr.shape)}")
        lines.append(" ".join(f"{x:.17e}" for x in arr.ravel()))
    with open(os.path.join(HERE, "tiny_causal_gqa.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
