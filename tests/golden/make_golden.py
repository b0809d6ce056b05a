"""Writes tests/golden/tiny_f32_oracle.json from the CPU oracle only.

Regression fixture for the oracle on the tiny fp32 workload
(batch 1, seqlen 256, 4 heads, headdim 16, d_state 16, 1 group, seed 0).
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from state_space_model_sm_gb300.inputs import SSDShape, make_inputs  # noqa: E402


def main():
    inp = make_inputs(SSDShape(1, 256, 4, 16, 16, 1, 64), seed=0, dtype="f32")
    y, final = oracle.ssd_fwd(*oracle.from_inputs(inp))
    samples = {}
    for (t, h, p) in [(0, 0, 0), (1, 2, 5), (63, 1, 15), (64, 3, 7), (200, 0, 9), (255, 3, 15)]:
        samples[f"{t},{h},{p}"] = float(y[0, t, h, p])
    out = dict(workload="tiny_f32 seed 0", y_samples=samples, y_sum=float(np.sum(y)),
               final_sq=float(np.sum(final ** 2)))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_f32_oracle.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
