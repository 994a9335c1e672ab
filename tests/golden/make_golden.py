"""Writes tiny_oracle_regression.json from the fp64 oracle alone.

The pages print no numeric worked example for the layer, so this fixture is a
regression record of the oracle itself on a tiny seeded case: any later change
to the oracle's arithmetic shows up as a diff here and must be justified.
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from dropless_mixture_experts_top_gb300 import synth  # noqa: E402
from oracle import oracle as O  # noqa: E402

SHAPE = synth.MoEShape(T=16, H=32, I=32, E=4, k=2)
SEED = 7


def compute():
    inp = synth.make_inputs_shape(SHAPE, SEED, w_scale=0.3)
    idx, w = O.route(inp["logits"], SHAPE.k)
    out = O.forward(SHAPE, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"])
    dx, dl, _ = O.backward_tokens(SHAPE, inp["x"], inp["logits"], idx, w, inp["W_gate"], inp["W_up"],
                                  inp["W_down"], inp["dy"])
    dWg, dWu, dWd = O.dw_full(SHAPE, inp["x"], idx, w, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"])
    counts, offsets, ros, sor = O.dispatch(idx, SHAPE.E)
    return {
        "shape": dict(T=SHAPE.T, H=SHAPE.H, I=SHAPE.I, E=SHAPE.E, k=SHAPE.k), "seed": SEED, "w_scale": 0.3,
        "topk_idx": idx.tolist(), "topk_w": w.tolist(), "counts": counts.tolist(),
        "row_of_slot": ros.tolist(),
        "out_rows0_3": out[:4].tolist(), "dx_rows0_3": dx[:4].tolist(), "d_logits": dl.tolist(),
        "dW_gate_e0_row0": dWg[0, 0].tolist(), "dW_up_e1_row5": dWu[1, 5].tolist(),
        "dW_down_e2_row3": dWd[2, 3].tolist(),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_regression.json")
    with open(path, "w") as f:
        json.dump(compute(), f, indent=0)
        f.write("\n")
    print("wrote", path)
