"""GPU parity of the final RMSNorm + LM head + cross-entropy chain (logits never stored)
against the fp64 oracle, through the C ABI.

The forward GEMM's epilogue keeps, per row and per 256-column vocabulary tile, the online
softmax state (max, sum-exp) and the target's logit; a light reduce combines the tiles into
the log-sum-exp and the loss ("CODA: new research optimizes Transformer training with
GEMM-epilogue programming", kucoin.com news flash, sections "El epílogo esconde un tesoro" and
"Cinco bloques y un lenguaje LEGO").  The backward recomputes the logits in the epilogue of
the same GEMM and emits e = r dloss (softmax - onehot) / M, then reuses the RMSNorm-backward
combine of the block chain."""
import numpy as np
import pytest
import torch

import coda_synth as S
import oracle as O
from tests.gpu_helpers import TOL_BF16, assert_close, dev, f64, fresh_status, seeded

pytestmark = pytest.mark.gpu
BF = torch.bfloat16
LLAMA3_VOCAB = 128256


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def normwise(got, ref):
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


def test_xent_partials_epilogue(C):
    M, K, V = 300, 256, 800          # V = 3 full 256-column tiles + a 32-column tail
    u = seeded((M, K), 70, dtype=BF)
    W = seeded((V, K), 71, std=0.2, dtype=BF)
    r = seeded((M,), 72, std=0.2, mean=1.0)
    tg = torch.randint(0, V, (M,), generator=torch.Generator().manual_seed(73), dtype=torch.int32)
    n = (V + 255) // 256
    Pm = torch.empty((n, M), device="cuda")
    Ps = torch.empty((n, M), device="cuda")
    T = torch.empty((M,), device="cuda")
    C.coda_gemm_epilogue(dev(u), dev(W), [C.OP_ROW_SCALE, C.OP_XENT_PARTIAL], None, out_shape=(M, V),
                         row_scale=dev(r), row_index=dev(tg), row_partials=Pm, row_partials2=Ps, row_values=T)
    torch.cuda.synchronize()
    fresh_status()
    z = f64(r)[:, None] * O.linear(f64(u), f64(W))
    m_ref, s_ref = O.xent_partials(z, 256)
    assert_close(f64(Pm), m_ref, TOL_BF16, "tile maxima")
    # sum-exp partials are relative to the GPU's own maxima: compare the combined lse
    assert_close(O.xent_combine(f64(Pm), f64(Ps)), O.logsumexp(z), 1e-4, "log-sum-exp from the partials")
    assert_close(f64(T), z[np.arange(M), tg.numpy()], TOL_BF16, "target logits")
    lse, loss = torch.empty((M,), device="cuda"), torch.empty((M,), device="cuda")
    mean = torch.empty((1,), device="cuda")
    C.coda_xent_combine(Pm, Ps, T, dev(tg), V, lse, loss, mean)
    torch.cuda.synchronize()
    ce = O.cross_entropy(z, tg.numpy())
    assert_close(f64(lse), ce["lse"], 1e-4, "lse")
    assert_close(f64(loss), ce["loss"], 1e-3, "loss")
    np.testing.assert_allclose(float(mean.item()), ce["mean"], rtol=1e-4)


def _run_fwd(C, inp):
    h, g, W, tg = (dev(inp[k]) for k in ("h", "g", "W_v", "targets"))
    M, H = h.shape
    V = W.shape[0]
    o = dict(u=torch.empty((M, H), dtype=BF, device="cuda"), r=torch.empty((M,), device="cuda"),
             lse=torch.empty((M,), device="cuda"), loss=torch.empty((M,), device="cuda"),
             mean=torch.empty((1,), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_XENT_FWD, M, H, V) // 4,), device="cuda")
    C.coda_lm_head_xent_forward(h, g, W, tg, inp["eps"], o["u"], o["r"], o["lse"], o["loss"], o["mean"], ws)
    torch.cuda.synchronize()
    fresh_status()
    return o, (h, g, W, tg)


def _run_bwd(C, fwd, dv, dloss):
    h, g, W, tg = dv
    M, H = h.shape
    V = W.shape[0]
    o = dict(e=torch.empty((M, V), dtype=BF, device="cuda"), dh=torch.empty((M, H), dtype=BF, device="cuda"),
             dW_v=torch.empty((V, H), device="cuda"), dg=torch.empty((H,), device="cuda"),
             c=torch.empty((M,), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_XENT_BWD, M, H, V) // 4,), device="cuda")
    C.coda_lm_head_xent_backward(h, g, W, tg, fwd["u"], fwd["r"], fwd["lse"], dloss, o["e"], o["dh"], o["dW_v"],
                                 o["dg"], o["c"], ws)
    torch.cuda.synchronize()
    fresh_status()
    return o


def test_lm_head_xent_uniform_logits_closed_form(C):
    """A zero LM head makes every logit 0: the loss of each row is log V, the gradient of the
    logits is r dloss (1/V - onehot) / M, and no gradient reaches h (c = 0, t = 0)."""
    M, H, V = 300, 256, 992
    inp = S.lm_head_inputs(M, H, V, seed=2)
    inp["W_v"] = torch.zeros_like(inp["W_v"])
    fwd, dv = _run_fwd(C, inp)
    np.testing.assert_allclose(f64(fwd["lse"]), np.log(V), rtol=1e-6)
    np.testing.assert_allclose(f64(fwd["loss"]), np.log(V), rtol=1e-6)
    np.testing.assert_allclose(float(fwd["mean"].item()), np.log(V), rtol=1e-6)
    dloss = 1.0
    bwd = _run_bwd(C, fwd, dv, dloss)
    r = f64(fwd["r"])
    onehot = np.zeros((M, V))
    onehot[np.arange(M), inp["targets"].numpy()] = 1.0
    e_ref = r[:, None] * dloss * (1.0 / V - onehot) / M
    assert_close(f64(bwd["e"]), e_ref, TOL_BF16, "e")
    assert not f64(bwd["dh"]).any(), "dh must be zero"
    assert not f64(bwd["c"]).any(), "c must be zero"


@pytest.mark.parametrize("M,H,V", [(300, 256, 992), (512, 512, 4096)])
def test_lm_head_xent_small(C, M, H, V):
    inp = S.lm_head_inputs(M, H, V, seed=1, w_std=0.1)
    fwd, dv = _run_fwd(C, inp)
    x = {k: f64(inp[k]) for k in ("h", "g", "W_v")}
    t = inp["targets"].numpy()
    ref = O.lm_head_xent_forward(x["h"], x["g"], x["W_v"], t, inp["eps"])
    assert_close(f64(fwd["r"]), ref["r"], TOL_BF16, "r")
    assert_close(f64(fwd["u"]), x["h"] * x["g"][None, :], TOL_BF16, "u = h g")
    assert_close(f64(fwd["lse"]), ref["lse"], TOL_BF16, "lse")
    assert_close(f64(fwd["loss"]), ref["loss"], TOL_BF16, "loss")
    np.testing.assert_allclose(float(fwd["mean"].item()), ref["mean"], rtol=2e-3)
    bwd = _run_bwd(C, fwd, dv, dloss=1.0)
    fused = O.lm_head_xent_backward_fused(ref, x["h"], x["g"], x["W_v"], t, 1.0)
    plain = O.lm_head_xent_backward(ref, x["h"], x["g"], x["W_v"], t, 1.0)
    # e is a difference of two nearly equal terms at the target column: hold it normwise
    assert normwise(f64(bwd["e"]), fused["e"]) <= TOL_BF16, "e"
    assert_close(f64(bwd["c"]), fused["c"], TOL_BF16, "c")
    for k in ("dh", "dg"):
        assert_close(f64(bwd[k]), plain[k], TOL_BF16, k)
    assert normwise(f64(bwd["dW_v"]), plain["dW_v"]) <= TOL_BF16, "dW_v"


@pytest.mark.slow
def test_lm_head_xent_full_size_sampled_rows(C):
    M, H, V = 16384, 2048, LLAMA3_VOCAB
    inp = S.lm_head_inputs(M, H, V, seed=0)
    fwd, dv = _run_fwd(C, inp)
    rows = np.sort(np.concatenate([np.arange(128), np.random.default_rng(5).choice(np.arange(128, M), 128,
                                                                                    replace=False)]))
    x = {k: f64(inp[k]) for k in ("h", "g", "W_v")}
    t = inp["targets"].numpy()
    ref = O.lm_head_xent_forward(x["h"][rows], x["g"], x["W_v"], t[rows], inp["eps"])
    assert_close(f64(fwd["lse"])[rows], ref["lse"], TOL_BF16, "lse rows")
    assert_close(f64(fwd["loss"])[rows], ref["loss"], TOL_BF16, "loss rows")
    # the mean is the fixed-order mean of every row's loss
    np.testing.assert_allclose(float(fwd["mean"].item()), float(np.mean(f64(fwd["loss"]))), rtol=1e-5)
    bwd = _run_bwd(C, fwd, dv, dloss=1.0)
    # row-local backward outputs on the sampled rows (the 1/M of the mean uses the full M)
    fused = O.lm_head_xent_backward_fused(ref, x["h"][rows], x["g"], x["W_v"], t[rows], dloss=len(rows) / M)
    assert normwise(f64(bwd["e"])[rows], fused["e"]) <= TOL_BF16, "e rows"
    assert_close(f64(bwd["c"])[rows], fused["c"], TOL_BF16, "c rows")
    assert_close(f64(bwd["dh"])[rows], fused["dh"], TOL_BF16, "dh rows")
