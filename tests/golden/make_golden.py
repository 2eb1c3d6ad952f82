"""Writes tests/golden/tiny_oracle.json: a regression fixture of the fp64
oracle on the seeded tiny workload (T=64, H=128, I=64, E=8, K=2).

It calls only the oracle and the seeded input generators.  The fixture guards
the oracle against unintended changes; its independent pins are the closed
forms, special cases and finite differences in tests/test_oracle_pins.py.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402
import oracle  # noqa: E402

SAMPLES = [(0, 0), (5, 17), (31, 127), (63, 64)]


def compute():
    p = mi.make("tiny")
    y = oracle.forward(p.x, p.topk_ids, p.topk_weights, p.W1, p.W2)
    dx, dW1, dW2, dw = oracle.backward(p.x, p.topk_ids, p.topk_weights, p.W1, p.W2, p.dy)
    counts, offsets, s2r, r2s = oracle.route(p.topk_ids, p.shape.E)
    return {
        "workload": "tiny: T=64 H=128 I=64 E=8 K=2, seed 1000, uniform distinct routing",
        "counts": counts.tolist(),
        "row2slot_head": r2s[:16].tolist(),
        "y": {f"{t},{c}": float(y[t, c]) for t, c in SAMPLES},
        "dx": {f"{t},{c}": float(dx[t, c]) for t, c in SAMPLES},
        "dw": {f"{t},{k}": float(dw[t, k]) for t, k in [(0, 0), (7, 1), (63, 1)]},
        "dW1": {f"{e},{i},{j}": float(dW1[e, i, j]) for e, i, j in [(0, 0, 0), (3, 100, 90), (7, 127, 127)]},
        "dW2": {f"{e},{i},{j}": float(dW2[e, i, j]) for e, i, j in [(0, 0, 0), (4, 33, 70), (7, 63, 127)]},
        "y_abs_sum": float(abs(y).sum()),
        "dW1_abs_sum": float(abs(dW1).sum()),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
    print("wrote", out)
