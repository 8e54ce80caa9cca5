"""GPU parity of the chains (tiny fp32 chain, LLaMA-shaped block forward / backward, QKV +
RoPE, fp8 MLP) against the fp64 oracle, through the C ABI.

Reduced sizes compare every output element; the full 16384-token sizes (the launch
configuration the bench times) compare sampled token rows (rows 0-255 plus 256 random
rows: forward rows are independent, so the oracle computes exactly those rows) and, for
weight gradients, sampled columns over all rows.

Tensors that are products of two bf16-stored GEMM results (a, e and the weight gradients
dW_d, dW_gu built from them) get two checks: against the oracle's plain chain (normwise,
and element-wise against the bf16-storage model), and element by element at 2e-2 against
the oracle given the chain's own stored inputs of that step (exact inputs: the u or h the
gate/up GEMM read, r, the saved Z, a, e, dh).  The second holds each kernel to the bar
wherever the chain stands, the first bounds how far bf16 storage moves the chain."""
import numpy as np
import pytest
import torch

import coda_synth as S
import oracle as O
from tests import storage_sim as SIM
from tests.gpu_helpers import (TOL_BF16, TOL_FP8, assert_close, assert_e4m3_codes, assert_product_close, dev, f64,
                               fresh_status)

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def sample_rows(M, seed=0):
    rng = np.random.default_rng(seed)
    extra = rng.choice(np.arange(256, M), size=min(256, max(M - 256, 0)), replace=False)
    return np.sort(np.concatenate([np.arange(min(256, M)), extra]))


# --------------------------------------------------------------------- tiny fp32 chain
def test_tiny_fp32_chain(C):
    t = S.tiny_chain_inputs()
    X, R, W1, W2, g = (t[k] for k in ("X", "R", "W1", "W2", "g"))
    M, d = X.shape
    n2 = W2.shape[1]
    W1t, W2t = dev(W1.t().contiguous()), dev(W2.t().contiguous())   # [out, in] weights
    h = torch.empty((M, d), dtype=torch.float32, device="cuda")
    P = torch.empty((1, M), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(X), W1t, [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL], h, residual=dev(R), row_partials=P)
    r = torch.empty((M,), dtype=torch.float32, device="cuda")
    C.coda_rms_partial_reduce(P, M, d, t["eps"], r)
    W2f = torch.empty_like(W2t)
    C.coda_fold_gain(W2t, dev(g), W2f)
    out = torch.empty((M, n2), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(h, W2f, [C.OP_ROW_SCALE], out, row_scale=r)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.tiny_chain(f64(X), f64(R), f64(W1), f64(W2), f64(g), t["eps"])
    assert_close(f64(h), ref["h"], TOL_BF16, "h")
    assert_close(f64(r), ref["r"], TOL_BF16, "r")
    assert_close(f64(out), ref["out"], TOL_BF16, "out")


# --------------------------------------------------------------------- block forward
def _run_block_forward(C, inp, train=True, gain="broadcast"):
    """gain = "broadcast": G1's epilogue stores u = h g and G2 reads it with the unfolded
    W_gu; gain = "fold": W_gu' = W_gu diag(g) first (coda_fold_gain) and G2 reads h."""
    O_, R, W_o, W_gu, W_d, g = (dev(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g"))
    M, H = O_.shape
    F = W_d.shape[1]
    out = dict(h=torch.empty((M, H), dtype=BF, device="cuda"), r=torch.empty((M,), device="cuda"),
               a=torch.empty((M, F), dtype=BF, device="cuda"), Y=torch.empty((M, H), dtype=BF, device="cuda"),
               Z=torch.empty((M, 2 * F), dtype=BF, device="cuda") if train else None,
               Yp=torch.empty(((H + 255) // 256, M), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    if gain == "fold":
        Wf = torch.empty_like(W_gu)
        C.coda_fold_gain(W_gu, g, Wf)
        out["Wf"] = Wf
        C.coda_block_forward(O_, R, W_o, Wf, W_d, inp["eps"], out["h"], out["r"], out["a"], out["Y"], ws,
                             Z=out["Z"], Y_partials=out["Yp"])
    else:
        out["u"] = torch.empty((M, H), dtype=BF, device="cuda")
        C.coda_block_forward(O_, R, W_o, W_gu, W_d, inp["eps"], out["h"], out["r"], out["a"], out["Y"], ws,
                             Z=out["Z"], Y_partials=out["Yp"], g=g, u=out["u"])
    torch.cuda.synchronize()
    fresh_status()
    return out, None


def _a_exact_inputs(out, inp, rows):
    """a on `rows` from the inputs the gate/up GEMM read in this chain: the stored bf16 u = h g
    with the unfolded W_gu (gain broadcast), or the stored h with the folded bf16 W_gu', and
    the chain's fp32 r:  Z = r (x W^T),  a = silu(G) U  (fp64)."""
    if "Wf" in out:
        x, W = f64(out["h"])[rows], f64(out["Wf"])
    else:
        x, W = f64(out["u"])[rows], f64(inp["W_gu"])
    Z = f64(out["r"])[rows][:, None] * O.linear(x, W)
    F = Z.shape[1] // 2
    return O.swiglu(Z[:, :F], Z[:, F:])


def _oracle_forward_rows(inp, rows):
    x = {k: f64(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    return O.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"])


def _sim_forward_rows(inp, rows, gain="broadcast"):
    x = {k: f64(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    return SIM.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"], gain)


def test_block_forward_zero_and_constant_rows(C):
    """Degenerate rows of the RMSNorm: a zero row of h (O and R zero) has r = (0 + eps)^(-1/2)
    exactly and zero outputs; rows where O W_o^T + R is zero but for one column keep r finite;
    the other rows are unaffected."""
    M, H, F = 300, 256, 384
    inp = S.block_inputs(M, H, F, seed=11)
    inp["O"][:4] = 0
    inp["R"][:4] = 0                                          # rows 0-3: h = 0
    inp["O"][4:6] = 0
    inp["R"][4:6] = 0
    inp["R"][4:6, 7] = 3.0                                   # rows 4, 5: h = 3 e_7
    out, _ = _run_block_forward(C, inp)
    eps = inp["eps"]
    r = f64(out["r"])
    np.testing.assert_allclose(r[:4], 1.0 / np.sqrt(eps), rtol=1e-6)
    np.testing.assert_allclose(r[4:6], 1.0 / np.sqrt(9.0 / H + eps), rtol=1e-6)   # one nonzero a: |a| / sqrt(d)
    assert not f64(out["Y"])[:4].any() and not f64(out["a"])[:4].any()
    ref = _oracle_forward_rows(inp, np.arange(M))
    assert_close(f64(out["Y"]), ref["Y"], TOL_BF16, "Y")
    assert_close(r, ref["r"], TOL_BF16, "r")


@pytest.mark.parametrize("gain", ["broadcast", "fold"])
@pytest.mark.parametrize("M,H,F", [(640, 512, 1024), (300, 256, 384)])
def test_block_forward_small(C, M, H, F, gain):
    _check_block_forward(C, M, H, F, gain)


# hidden sizes of the 7B and 70B LLaMA-3 shapes (the pages' 1B / 7B / 70B sweep), fewer tokens
@pytest.mark.parametrize("M,H,F", [(256, 4096, 14336), (128, 8192, 28672)])
def test_block_forward_7b_70b_hidden_sizes(C, M, H, F):
    _check_block_forward(C, M, H, F, "broadcast")


def _check_block_forward(C, M, H, F, gain):
    inp = S.block_inputs(M, H, F, seed=0)
    out, _ = _run_block_forward(C, inp, gain=gain)
    ref = _oracle_forward_rows(inp, np.arange(M))
    sim = _sim_forward_rows(inp, np.arange(M), gain)
    for k in ("h", "r", "Y"):
        assert_close(f64(out[k]), ref[k], TOL_BF16, k)
    assert_product_close(f64(out["a"]), ref["a"], sim["a"], "a")
    assert_close(f64(out["a"]), _a_exact_inputs(out, inp, np.arange(M)), TOL_BF16, "a (exact inputs)")
    assert_close(f64(out["Z"]), ref["Z"], TOL_BF16, "Z")
    assert_close(f64(out["Yp"]), O.partial_sumsq(ref["Y"], 256), TOL_BF16, "Y partials")
    if gain == "broadcast":
        assert_close(f64(out["u"]), ref["h"] * f64(inp["g"])[None, :], TOL_BF16, "u = h g")


@pytest.mark.slow
def test_block_forward_full_size_sampled_rows(C):
    M, H, F = 16384, 2048, 8192
    inp = S.block_inputs(M, H, F, seed=0)
    out, _ = _run_block_forward(C, inp, train=False)
    rows = sample_rows(M)
    ref = _oracle_forward_rows(inp, rows)
    sim = _sim_forward_rows(inp, rows)
    for k in ("h", "r", "Y"):
        assert_close(f64(out[k])[rows], ref[k], TOL_BF16, k)
    assert_product_close(f64(out["a"])[rows], ref["a"], sim["a"], "a")
    assert_close(f64(out["a"])[rows], _a_exact_inputs(out, inp, rows), TOL_BF16, "a (exact inputs)")


# --------------------------------------------------------------------- block backward
def _run_block_backward(C, inp, fwd_out):
    O_, W_o, W_gu, W_d, g, dY = (dev(inp[k]) for k in ("O", "W_o", "W_gu", "W_d", "g", "dY"))
    M, H = O_.shape
    F = W_d.shape[1]
    o = dict(e=torch.empty((M, 2 * F), dtype=BF, device="cuda"), dh=torch.empty((M, H), dtype=BF, device="cuda"),
             dO=torch.empty((M, H), dtype=BF, device="cuda"), dW_o=torch.empty((H, H), device="cuda"),
             dW_gu=torch.empty((2 * F, H), device="cuda"), dW_d=torch.empty((H, F), device="cuda"),
             dg=torch.empty((H,), device="cuda"), c=torch.empty((M,), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_BWD, M, H, F) // 4,), device="cuda")
    C.coda_block_backward(O_, W_o, W_gu, W_d, g, fwd_out["h"], fwd_out["r"], fwd_out["Z"], fwd_out["a"], dY,
                          o["e"], o["dh"], o["dO"], o["dW_o"], o["dW_gu"], o["dW_d"], o["dg"], o["c"], ws)
    torch.cuda.synchronize()
    fresh_status()
    return o


def _e_exact_inputs(fwd, inp, rows):
    """e on `rows` from the saved bf16 Z = [G | U], the chain's r and dY (fp64):
    dA = dY W_d,  e = r [dA U silu'(G) | dA silu(G)]."""
    Z, r = f64(fwd["Z"])[rows], f64(fwd["r"])[rows]
    dA = f64(inp["dY"])[rows] @ f64(inp["W_d"])
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    return r[:, None] * np.hstack([dA * U * O.silu_grad(G), dA * O.silu(G)])


def _check_backward_exact_inputs(inp, fwd, got, rows, fcols, hcols):
    """Each backward output against the oracle given the chain's own stored tensors: e on
    `rows`; dW_d[:, fcols] = dY^T a; dW_gu on the gate and up rows fcols, F + fcols as
    g (e^T h); dW_o[:, hcols] = dh^T O; dg[hcols] = sum_i h (e W_gu)[:, hcols]."""
    F = f64(inp["W_d"]).shape[1]
    assert_close(f64(got["e"])[rows], _e_exact_inputs(fwd, inp, rows), TOL_BF16, "e (exact inputs)")
    dY, Ox, g = f64(inp["dY"]), f64(inp["O"]), f64(inp["g"])
    h, a = f64(fwd["h"]), f64(fwd["a"])
    assert_close(f64(got["dW_d"])[:, fcols], dY.T @ a[:, fcols], TOL_BF16, "dW_d[:, cols] (exact inputs)")
    e_t = got["e"].cpu()
    ecols = np.concatenate([fcols, F + fcols])
    ref_dWgu = g[None, :] * (f64(e_t[:, torch.from_numpy(ecols)]).T @ h)
    assert_close(f64(got["dW_gu"])[ecols], ref_dWgu, TOL_BF16, "dW_gu[cols] (exact inputs)")
    assert_close(f64(got["dW_o"])[:, hcols], f64(got["dh"]).T @ Ox[:, hcols], TOL_BF16, "dW_o[:, cols] (exact inputs)")
    Wc = f64(inp["W_gu"])[:, hcols]
    dg = np.zeros(len(hcols))
    for i0 in range(0, h.shape[0], 2048):                       # t = e W_gu on the sampled columns
        dg += np.sum(h[i0:i0 + 2048, hcols] * (f64(e_t[i0:i0 + 2048]) @ Wc), axis=0)
    assert_close(f64(got["dg"])[hcols], dg, TOL_BF16, "dg[cols] (exact inputs)")


def test_block_backward_zero_output_gradient(C):
    """dY = 0: every gradient of the block is exactly zero (nothing stale from the workspace,
    the partial buffers or a previous call leaks in); the buffers start non-zero."""
    M, H, F = 300, 256, 384
    inp = S.block_inputs(M, H, F, seed=12, with_grad=True)
    fwd, _ = _run_block_forward(C, inp)
    warm = _run_block_backward(C, inp, fwd)                  # a call with a real dY first
    assert f64(warm["dh"]).any()
    inp["dY"] = torch.zeros_like(inp["dY"])
    o = _run_block_backward(C, inp, fwd)
    for k in ("e", "dh", "dO", "dW_o", "dW_gu", "dW_d", "dg", "c"):
        assert not f64(o[k]).any(), k


@pytest.mark.parametrize("M,H,F", [(640, 512, 1024), (300, 256, 384)])
def test_block_backward_small(C, M, H, F):
    inp = S.block_inputs(M, H, F, seed=0, with_grad=True)
    fwd, _ = _run_block_forward(C, inp)
    got = _run_block_backward(C, inp, fwd)
    x = {k: f64(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    ref_f = O.block_forward(x["O"], x["R"], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"])
    ref = O.block_backward(ref_f, x["O"], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"])
    fused = O.block_backward_fused(ref_f, x["O"], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"])
    sf = SIM.block_forward(x["O"], x["R"], x["W_o"], x["g"], x["W_gu"], x["W_d"], inp["eps"])
    sb = SIM.block_backward(sf, x["O"], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"])
    assert_product_close(f64(got["e"]), fused["e"], sb["e"], "e")
    assert_close(f64(got["c"]), fused["c"], TOL_BF16, "c")
    for k in ("dh", "dO", "dW_o", "dg"):
        assert_close(f64(got[k]), ref[k], TOL_BF16, k)
    for k in ("dW_gu", "dW_d"):
        assert_product_close(f64(got[k]), ref[k], sb[k], k)
    _check_backward_exact_inputs(inp, fwd, got, np.arange(M), np.arange(F), np.arange(H))


@pytest.mark.slow
def test_block_backward_full_size_sampled(C):
    M, H, F = 16384, 2048, 8192
    inp = S.block_inputs(M, H, F, seed=0, with_grad=True)
    fwd, _ = _run_block_forward(C, inp)
    got = _run_block_backward(C, inp, fwd)
    x = {k: f64(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    eps = inp["eps"]
    # row-local outputs on sampled rows
    rows = sample_rows(M, seed=1)
    rf = O.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], eps)
    rb = O.block_backward_fused(rf, x["O"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"][rows])
    sf = SIM.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], eps)
    sb = SIM.block_backward(sf, x["O"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"][rows])
    for k in ("dh", "dO", "c"):
        assert_close(f64(got[k])[rows], rb[k], TOL_BF16, k)
    assert_product_close(f64(got["e"])[rows], rb["e"], sb["e"], "e")
    # weight gradients on sampled columns, summed over all rows (oracle, and the bf16-storage
    # model of the same columns)
    cols = np.sort(np.random.default_rng(2).choice(F, size=64, replace=False))
    dA = x["dY"] @ x["W_d"][:, cols]
    h = O.linear(x["O"], x["W_o"]) + x["R"]
    r = O.rms_scale(h, eps)
    Wf = O.fold_gain(x["W_gu"], x["g"])
    G, U = r[:, None] * (h @ Wf[cols].T), r[:, None] * (h @ Wf[F + cols].T)
    ref_dWd = x["dY"].T @ O.swiglu(G, U)
    ref_dWgu = x["g"][None, :] * ((r[:, None] * dA * U * O.silu_grad(G)).T @ h)
    hs = SIM.bf(h)
    rs = SIM.f32(1.0 / np.sqrt(np.mean(hs * hs, axis=1) + eps))
    Wfs = SIM.bf(Wf)
    Gs, Us = SIM.bf(rs[:, None] * (hs @ Wfs[cols].T)), SIM.bf(rs[:, None] * (hs @ Wfs[F + cols].T))
    sim_dWd = x["dY"].T @ SIM.bf(O.swiglu(Gs, Us))
    sim_dWgu = x["g"][None, :] * (SIM.bf(rs[:, None] * dA * Us * O.silu_grad(Gs)).T @ hs)
    assert_product_close(f64(got["dW_d"])[:, cols], ref_dWd, sim_dWd, "dW_d[:, cols]")
    assert_product_close(f64(got["dW_gu"])[cols], ref_dWgu, sim_dWgu, "dW_gu[cols]")
    # every output, dW_o and dg included, against the oracle given the chain's stored tensors
    hcols = np.sort(np.random.default_rng(6).choice(H, size=64, replace=False))
    _check_backward_exact_inputs(inp, fwd, got, rows, cols, hcols)


# --------------------------------------------------------------------- QKV + RoPE
def _run_qkv(C, inp, seq, hd, n_rot):
    h, W, g = dev(inp["h"]), dev(inp["W_qkv"]), dev(inp["g"])
    M, H = h.shape
    N = W.shape[0]
    Wf = torch.empty_like(W)
    C.coda_fold_gain(W, g, Wf)
    cos = torch.empty((seq, hd // 2), device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, 500000.0, cos, sin)
    r = torch.empty((M,), device="cuda")
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_qkv_rope(h, Wf, inp["eps"], seq, hd, n_rot, cos, sin, r, out)
    torch.cuda.synchronize()
    fresh_status()
    return out, r


def test_qkv_rope_small(C):
    M, H, seq, hd = 512, 256, 128, 64
    inp = S.qkv_inputs(M, H, (4 + 2 * 2) * hd, seed=0)
    out, r = _run_qkv(C, inp, seq, hd, (4 + 2) * hd)
    ref = O.qkv_rope(f64(inp["h"]), f64(inp["g"]), f64(inp["W_qkv"]), inp["eps"], seq, (4 + 2) * hd, hd, 500000.0)
    assert_close(f64(r), ref["r"], TOL_BF16, "r")
    assert_close(f64(out), ref["out"], TOL_BF16, "qkv")


def test_qkv_rope_ragged_rows_every_row(C):
    """3300 tokens (a ragged last tile of 228 rows, RoPE positions wrapping at 1024) x 3072
    columns: every row is checked against the oracle."""
    M, H, seq, hd = 3300, 256, 1024, 64
    inp = S.qkv_inputs(M, H, 3072, seed=4)
    out, r = _run_qkv(C, inp, seq, hd, 2560)
    ref = O.qkv_rope(f64(inp["h"]), f64(inp["g"]), f64(inp["W_qkv"]), inp["eps"], seq, 2560, hd, 500000.0)
    assert_close(f64(r), ref["r"], TOL_BF16, "r")
    assert_close(f64(out), ref["out"], TOL_BF16, "qkv")
    assert_close(f64(out)[3072:], ref["out"][3072:], TOL_BF16, "qkv, rows of the last tile")


@pytest.mark.slow
def test_qkv_rope_full_size_sampled_rows(C):
    M, H, seq, hd = 16384, 2048, 1024, 64
    inp = S.qkv_inputs(M, H, 3072, seed=0)
    out, r = _run_qkv(C, inp, seq, hd, 2560)
    rows = np.union1d(sample_rows(M, seed=3), np.arange(M - 64, M))   # and rows of the last block
    hq = f64(inp["h"])[rows]
    y = O.rmsnorm(hq, f64(inp["g"]), inp["eps"]) @ f64(inp["W_qkv"]).T
    ref = O.rope_rotate(y, rows % seq, 2560, hd, 500000.0)
    assert_close(f64(out)[rows], ref, TOL_BF16, "qkv rows")


@pytest.mark.parametrize("M", [1, 7, 1000, 1001, 16384])
def test_chain_row_rms_bitwise_equal_to_row_rms(C, M):
    """The QKV + RoPE chain and the FP8 MLP open with a one-CTA-per-SM row RMS that shares the
    standalone pass's summation order: r must be the same bits as coda_row_rms gives for the
    same h, for row counts below one warp's group of 4 rows, ragged, and full size (every
    SM's CTA taking several groups)."""
    H, hd = 2048, 64
    inp = S.qkv_inputs(M, H, 8 * hd, seed=5)
    _, r_chain = _run_qkv(C, inp, 128, hd, 6 * hd)
    r_plain = torch.empty((M,), device="cuda")
    C.coda_row_rms(dev(inp["h"]), inp["eps"], r_plain)
    torch.cuda.synchronize()
    fresh_status()
    assert torch.equal(r_chain, r_plain)
    if M < 1000:
        return   # the FP8 chain at the larger row counts (ragged and not) only
    fi = S.fp8_mlp_inputs(M, 512, 384, seed=5)
    r8 = _run_fp8(C, fi, 1.0)[0]
    r8_plain = torch.empty((M,), device="cuda")
    C.coda_row_rms(dev(fi["h"]), fi["eps"], r8_plain)
    torch.cuda.synchronize()
    fresh_status()
    assert torch.equal(r8, r8_plain)


# --------------------------------------------------------------------- FP8 MLP
def _run_fp8(C, inp, s_a):
    h, Xq, Wq, Wdq = dev(inp["h"]), dev(inp["Xq"]), dev(inp["Wq"]), dev(inp["Wdq"])
    M, H = h.shape
    F = Wdq.shape[1]
    r = torch.empty((M,), device="cuda")
    aq = torch.empty((M, F), dtype=torch.uint8, device="cuda")
    amax = torch.empty((1,), device="cuda")
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty(((H + 255) // 256, M), device="cuda")
    C.coda_mlp_fp8(h, Xq, Wq, Wdq, inp["s_x"], inp["s_w"], inp["s_wd"], s_a, inp["eps"], r, aq, amax, Y, P)
    torch.cuda.synchronize()
    fresh_status()
    return r, aq, amax, Y, P


def _fp8_oracle(inp, rows, s_a):
    return O.mlp_fp8(f64(inp["h"])[rows], f64(inp["Xq"])[rows], inp["s_x"], f64(inp["Wq"]), inp["s_w"],
                     f64(inp["Wdq"]), inp["s_wd"], s_a, inp["eps"], 256)


def _fp8_checks(inp, rows, r, aq, Y, P, s_a, ref):
    assert_close(f64(r)[rows], ref["r"], TOL_BF16, "r")
    assert_e4m3_codes(aq.cpu().numpy()[rows], ref["a"] / s_a, "a_q codes")
    assert_close(f64(Y)[rows], ref["Y"], TOL_FP8, "Y")
    assert_close(f64(P)[:, rows], ref["P"], TOL_FP8, "Y partials")


@pytest.mark.parametrize("M,H,F", [(512, 512, 768), (300, 256, 384)])   # the second ragged in M and in tiles
def test_fp8_mlp_small(C, M, H, F):
    inp = S.fp8_mlp_inputs(M, H, F, seed=0)
    rows = np.arange(M)
    s_a = float(_fp8_oracle(inp, rows, 1.0)["amax"]) / 448.0   # delayed scaling from a prior pass
    r, aq, amax, Y, P = _run_fp8(C, inp, s_a)
    ref = _fp8_oracle(inp, rows, s_a)
    _fp8_checks(inp, rows, r, aq, Y, P, s_a, ref)
    np.testing.assert_allclose(float(amax.item()), ref["amax"], rtol=2e-2)


@pytest.mark.slow
def test_fp8_mlp_full_size_sampled_rows(C):
    M, H, F = 16384, 4096, 14336
    inp = S.fp8_mlp_inputs(M, H, F, seed=0)
    rows = sample_rows(M, seed=4)
    s_a = 4.0 * float(_fp8_oracle(inp, rows[:64], 1.0)["amax"]) / 448.0
    r, aq, amax, Y, P = _run_fp8(C, inp, s_a)
    ref = _fp8_oracle(inp, rows, s_a)
    _fp8_checks(inp, rows, r, aq, Y, P, s_a, ref)
    assert float(amax.item()) >= ref["amax"] * (1 - 2e-2)
