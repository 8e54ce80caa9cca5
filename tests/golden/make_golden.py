"""Writes the oracle regression fixtures in this folder.  Calls only the oracle (and numpy
for the seeded inputs, which are stored in the fixture beside the outputs).

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle as O  # noqa: E402


def tiny_block():
    rng = np.random.default_rng(20260522)
    M, d, F = 3, 8, 4
    inp = dict(O=rng.normal(size=(M, d)), R=rng.normal(size=(M, d)),
               W_o=rng.normal(size=(d, d)) / 3, g=1 + 0.1 * rng.normal(size=d),
               W_gu=rng.normal(size=(2 * F, d)) / 3, W_d=rng.normal(size=(d, F)) / 3,
               dY=rng.normal(size=(M, d)))
    inp = {k: np.round(v, 6) for k, v in inp.items()}   # short decimal text, exact in the file
    eps = 1e-6
    fwd = O.block_forward(inp["O"], inp["R"], inp["W_o"], inp["g"], inp["W_gu"], inp["W_d"], eps)
    bwd = O.block_backward(fwd, inp["O"], inp["W_o"], inp["g"], inp["W_gu"], inp["W_d"], inp["dY"])
    q = O.qkv_rope(inp["O"], inp["g"], np.vstack([inp["W_o"], inp["W_o"]]), eps, seq_len=2,
                   n_rot_cols=8, head_dim=4, base=500000.0)
    out = {k: fwd[k] for k in ("h", "r", "a", "Y")}
    out.update({k: bwd[k] for k in ("dh", "dO", "dW_o", "dg", "dW_gu", "dW_d")})
    out["qkv_rope"] = q["out"]
    tgt = np.array([1, 7, 3])
    ce = O.lm_head_xent_forward(inp["O"], inp["g"], inp["W_gu"], tgt, eps)
    ceb = O.lm_head_xent_backward(ce, inp["O"], inp["g"], inp["W_gu"], tgt)
    out["xent_loss"] = ce["loss"]
    out["xent_dh"] = ceb["dh"]
    return dict(eps=eps, inputs={k: v.tolist() for k, v in inp.items()},
                outputs={k: np.asarray(v).tolist() for k, v in out.items()})


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_block_oracle.json"), "w") as f:
        json.dump(tiny_block(), f, indent=1)
    print("wrote tiny_block_oracle.json")
