"""GPU parity of the QKV + RoPE backward (rotation transposed, attention-input RMSNorm
backward) against the fp64 oracle's plain chain rule, through the C ABI.

The forward of this path is the QKV projection with the deferred r and the RoPE epilogue
("CODA: new research optimizes Transformer training with GEMM-epilogue programming",
kucoin.com news flash, "El epílogo esconde un tesoro": RoPE rewritten as an epilogue, and
the backward inherits the structure)."""
import numpy as np
import pytest
import torch

import coda_synth as S
import oracle as O
from tests.gpu_helpers import TOL_BF16, assert_close, dev, f64, fresh_status, seeded

pytestmark = pytest.mark.gpu
BF = torch.bfloat16
BASE = 500000.0


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def _run(C, M, H, N, seq, hd, n_rot, seed):
    inp = S.qkv_inputs(M, H, N, seed=seed)
    h, W, g = (dev(inp[k]) for k in ("h", "W_qkv", "g"))
    dout = dev(seeded((M, N), seed + 100, dtype=BF))
    cos = torch.empty((seq, hd // 2), device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, BASE, cos, sin)
    Wf = torch.empty_like(W)
    C.coda_fold_gain(W, g, Wf)
    r = torch.empty((M,), device="cuda")
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_qkv_rope(h, Wf, inp["eps"], seq, hd, n_rot, cos, sin, r, out)
    o = dict(e=torch.empty((M, N), dtype=BF, device="cuda"), dh=torch.empty((M, H), dtype=BF, device="cuda"),
             dW=torch.empty((N, H), device="cuda"), dg=torch.empty((H,), device="cuda"),
             c=torch.empty((M,), device="cuda"))
    ws = torch.empty((((M + 31) // 32) * H,), device="cuda")
    C.coda_qkv_rope_backward(h, g, W, r, out, dout, seq, hd, n_rot, cos, sin, o["e"], o["dh"], o["dW"], o["dg"],
                             o["c"], ws)
    torch.cuda.synchronize()
    fresh_status()
    return inp, dout, o


@pytest.mark.parametrize("M,H,heads_q,heads_kv,seq", [(512, 256, 4, 2, 128), (300, 512, 8, 2, 100)])
def test_qkv_rope_backward_small(C, M, H, heads_q, heads_kv, seq):
    hd = 64
    N, n_rot = (heads_q + 2 * heads_kv) * hd, (heads_q + heads_kv) * hd
    inp, dout, got = _run(C, M, H, N, seq, hd, n_rot, seed=2)
    x = {k: f64(inp[k]) for k in ("h", "W_qkv", "g")}
    kw = dict(seq_len=seq, n_rot_cols=n_rot, head_dim=hd, base=BASE)
    plain = O.qkv_rope_backward(x["h"], x["g"], x["W_qkv"], f64(dout), inp["eps"], **kw)
    fwd = O.qkv_rope(x["h"], x["g"], x["W_qkv"], inp["eps"], **kw)
    fused = O.qkv_rope_backward_fused(x["h"], x["g"], x["W_qkv"], f64(dout), fwd["out"], inp["eps"], **kw)
    assert_close(f64(got["e"]), fused["e"], TOL_BF16, "e = r R(-phi) dout")
    assert_close(f64(got["c"]), fused["c"], TOL_BF16, "c")
    assert_close(f64(got["dh"]), plain["dh"], TOL_BF16, "dh")
    assert_close(f64(got["dg"]), plain["dg"], TOL_BF16, "dg")
    assert_close(f64(got["dW"]), plain["dW"], TOL_BF16, "dW_qkv")


@pytest.mark.slow
def test_qkv_rope_backward_full_size_sampled_rows(C):
    M, H, N, seq, hd, n_rot = 16384, 2048, 3072, 1024, 64, 2560
    inp, dout, got = _run(C, M, H, N, seq, hd, n_rot, seed=0)
    rows = np.sort(np.concatenate([np.arange(256), np.random.default_rng(6).choice(np.arange(256, M), 256,
                                                                                    replace=False)]))
    x = {k: f64(inp[k]) for k in ("h", "W_qkv", "g")}
    hr, dr = x["h"][rows], f64(dout)[rows]
    r = O.rms_scale(hr, inp["eps"])
    pos = rows % seq
    Z = r[:, None] * ((hr * x["g"][None, :]) @ x["W_qkv"].T)
    out = O.rope_rotate(Z, pos, n_rot, hd, BASE)
    e = r[:, None] * O.rope_rotate(dr, -pos, n_rot, hd, BASE)
    c = r * (r * np.sum(dr * out, axis=1)) / H
    dh = x["g"][None, :] * (e @ x["W_qkv"]) - c[:, None] * hr
    assert_close(f64(got["e"])[rows], e, TOL_BF16, "e rows")
    assert_close(f64(got["c"])[rows], c, TOL_BF16, "c rows")
    assert_close(f64(got["dh"])[rows], dh, TOL_BF16, "dh rows")
