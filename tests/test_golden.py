"""Regression pin: the oracle reproduces the committed tiny-block fixture (written by
tests/golden/make_golden.py from the oracle itself)."""
import json
import os

import numpy as np

import oracle as O

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_block_fixture():
    with open(os.path.join(HERE, "tiny_block_oracle.json")) as f:
        fx = json.load(f)
    i = {k: np.array(v) for k, v in fx["inputs"].items()}
    eps = fx["eps"]
    fwd = O.block_forward(i["O"], i["R"], i["W_o"], i["g"], i["W_gu"], i["W_d"], eps)
    bwd = O.block_backward(fwd, i["O"], i["W_o"], i["g"], i["W_gu"], i["W_d"], i["dY"])
    q = O.qkv_rope(i["O"], i["g"], np.vstack([i["W_o"], i["W_o"]]), eps, seq_len=2,
                   n_rot_cols=8, head_dim=4, base=500000.0)
    got = {k: fwd[k] for k in ("h", "r", "a", "Y")}
    got.update({k: bwd[k] for k in ("dh", "dO", "dW_o", "dg", "dW_gu", "dW_d")})
    got["qkv_rope"] = q["out"]
    tgt = np.array([1, 7, 3])
    ce = O.lm_head_xent_forward(i["O"], i["g"], i["W_gu"], tgt, eps)
    got["xent_loss"] = ce["loss"]
    got["xent_dh"] = O.lm_head_xent_backward(ce, i["O"], i["g"], i["W_gu"], tgt)["dh"]
    for k, v in fx["outputs"].items():
        np.testing.assert_allclose(got[k], np.array(v), rtol=1e-12, atol=1e-14, err_msg=k)
