"""Writes the stored expected values under tests/golden/ from the CPU oracle.

Run from the repository root:  python tests/golden/make_golden.py

The pages print no worked example for the anchor-attention forward, so the stored values
are oracle outputs on seeded inputs from ``gen``; they pin the oracle against drift
(a change of its arithmetic, or of the C compiler/libm on another host) and give the
GPU tests a fixed expectation for the smallest workload.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import gen  # noqa: E402
import oracle  # noqa: E402

ROWS = [0, 1, 2, 97, 128, 195]


def main() -> None:
    w = gen.WORKLOADS["vit14_f32"]
    x = gen.make_inputs(w, seed=0)
    Q = gen.to_float64(x["Q"], w.dtype)
    U = gen.to_float64(x["U"], w.dtype)
    V = gen.to_float64(x["V"], w.dtype)
    H = oracle.forward(Q, U, V, w.scale)
    doc = {
        "what": "oracle H rows of the smallest workload (B=1 heads=1 n=196 m=16 d=64, fp32 inputs, seed 0)",
        "source": "anchor-attention forward H = A Delta^-1 A^T V, AnchorFormer (arXiv 2505.16463); "
                  "values written by tests/golden/make_golden.py from oracle/",
        "workload": w.name,
        "seed": 0,
        "scale": w.scale,
        "input_fingerprint": {
            "Q_sum": float(Q.sum()), "U_sum": float(U.sum()), "V_sum": float(V.sum()),
            "Q_first": [float(v) for v in Q.reshape(-1)[:4]],
            "V_last": [float(v) for v in V.reshape(-1)[-4:]],
        },
        "rows": ROWS,
        "H_rows": [[float(v) for v in H[0, 0, r]] for r in ROWS],
        "H_sum": float(H.sum()),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "vit14_f32_seed0.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
