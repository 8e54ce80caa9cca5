"""GPU parity of the FP8 MLP's training path against the fp64 oracle, through the C ABI:
the e4m3 quantiser, the forward that saves Z = [G | U], and the backward (e4m3 operands
with MN-major descriptors, the SwiGLU backward with an e4m3 output and its amax, the
RMSNorm-backward combine without a gain).

At the reduced size both sides get the same saved tensors (the oracle's Z rounded to bf16,
its a_q codes and its r in fp32), so only accumulation order and e4m3 decisions near a
rounding midpoint separate them.  At the full size (16384 tokens, LLaMA-3-8B MLP) the GPU
backward runs on the GPU forward's outputs and is compared end to end on sampled rows and
columns."""
import numpy as np
import pytest
import torch

import coda_synth as S
import oracle as O
from tests import storage_sim as SIM
from tests.gpu_helpers import TOL_BF16, TOL_FP8, assert_close, assert_e4m3_codes, dev, f64, fresh_status
from tests.storage_sim import normwise

pytestmark = pytest.mark.gpu
BF = torch.bfloat16
U8 = torch.uint8


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def _fp32_codes(x, scale):
    """e4m3 codes of x * (1 / scale) with the product taken in fp32: the decision the
    quantiser makes, taken in the same precision."""
    inv = np.float32(1.0) / np.float32(scale)
    v = (np.asarray(x, np.float32) * inv).astype(np.float64)
    return O.e4m3_encode(v)


# ------------------------------------------------------------------------- quantiser
def test_quantize_e4m3_bit_exact_ragged_with_saturation_and_zeros(C):
    M, N = 300, 272
    g = torch.Generator().manual_seed(21)
    X = (torch.randn((M, N), generator=g) * 3.0)
    X[0, :8] = 0.0
    X[1, :8] = -0.0
    X[2, :4] = torch.tensor([1e4, -1e4, 3e3, -5e2])      # beyond 448 * scale: saturate
    X = X.to(BF)
    scale = 0.0137
    Q = torch.empty((M, N), dtype=U8, device="cuda")
    amax = torch.zeros((1,), device="cuda")
    C.coda_quantize_e4m3(dev(X), scale, Q, amax)
    torch.cuda.synchronize()
    fresh_status()
    np.testing.assert_array_equal(Q.cpu().numpy(), _fp32_codes(f64(X), scale))
    assert float(amax.item()) == float(np.max(np.abs(f64(X))))


def test_quantize_e4m3_strided_rows_and_empty(C):
    M, N, ld = 64, 48, 80
    g = torch.Generator().manual_seed(22)
    base = torch.randn((M, ld), generator=g).to(BF)
    X = dev(base)[:, :N]                                  # row stride 80
    Qbuf = torch.zeros((M, 64), dtype=U8, device="cuda")
    Q = Qbuf[:, :N]
    C.coda_quantize_e4m3(X, 0.01, Q)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Q.cpu().numpy(), _fp32_codes(f64(base[:, :N]), 0.01))
    assert np.all(Qbuf[:, N:].cpu().numpy() == 0)        # nothing written past the row
    E = torch.empty((0, N), dtype=BF, device="cuda")
    C.coda_quantize_e4m3(E, 0.01, torch.empty((0, N), dtype=U8, device="cuda"))


# ------------------------------------------------------------------- forward saving Z
def _forward(C, inp, s_a, save_Z=True):
    h, Xq, Wq, Wdq = dev(inp["h"]), dev(inp["Xq"]), dev(inp["Wq"]), dev(inp["Wdq"])
    M, H = h.shape
    F = Wdq.shape[1]
    out = dict(r=torch.empty((M,), device="cuda"), aq=torch.empty((M, F), dtype=U8, device="cuda"),
               amax=torch.empty((1,), device="cuda"), Y=torch.empty((M, H), dtype=BF, device="cuda"),
               P=torch.empty(((H + 255) // 256, M), device="cuda"),
               Z=torch.empty((M, 2 * F), dtype=BF, device="cuda") if save_Z else None)
    C.coda_mlp_fp8(h, Xq, Wq, Wdq, inp["s_x"], inp["s_w"], inp["s_wd"], s_a, inp["eps"], out["r"], out["aq"],
                   out["amax"], out["Y"], out["P"], Z=out["Z"])
    torch.cuda.synchronize()
    fresh_status()
    return out


def _oracle_fwd(inp, s_a, rows=None):
    rows = np.arange(inp["h"].shape[0]) if rows is None else rows
    return O.mlp_fp8(f64(inp["h"])[rows], f64(inp["Xq"])[rows], inp["s_x"], f64(inp["Wq"]), inp["s_w"],
                     f64(inp["Wdq"]), inp["s_wd"], s_a, inp["eps"], 256)


def test_fp8_forward_saves_Z_and_keeps_its_outputs(C):
    M, H, F = 384, 512, 768
    inp = S.fp8_mlp_inputs(M, H, F, seed=0)
    s_a = float(_oracle_fwd(inp, 1.0)["amax"]) / 448.0
    with_z = _forward(C, inp, s_a, True)
    without = _forward(C, inp, s_a, False)
    ref = _oracle_fwd(inp, s_a)
    assert_close(f64(with_z["Z"]), ref["Z"], TOL_BF16, "saved Z")
    for k in ("r", "aq", "Y", "P"):                       # saving Z changes nothing else
        assert torch.equal(with_z[k], without[k]), k


# --------------------------------------------------------------------------- backward
def _backward(C, inp, Z, aq, r, s_a, s_dy, s_e):
    h, Xq, Wq, Wdq, dY = (dev(inp[k]) for k in ("h", "Xq", "Wq", "Wdq", "dY"))
    M, H = h.shape
    F = Wdq.shape[1]
    o = dict(dYq=torch.empty((M, H), dtype=U8, device="cuda"), amax_dy=torch.empty((1,), device="cuda"),
             eq=torch.empty((M, 2 * F), dtype=U8, device="cuda"), amax_e=torch.empty((1,), device="cuda"),
             c=torch.empty((M,), device="cuda"), dh=torch.empty((M, H), dtype=BF, device="cuda"),
             dW_d=torch.empty((H, F), device="cuda"), dW=torch.empty((2 * F, H), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_MLP_FP8_BWD, M, H, F) // 4,), device="cuda")
    C.coda_mlp_fp8_backward(h, Xq, Wq, Wdq, Z, aq, r, dY, inp["s_x"], inp["s_w"], inp["s_wd"], s_a, s_dy, s_e,
                            o["dYq"], o["amax_dy"], o["eq"], o["amax_e"], o["c"], o["dh"], o["dW_d"], o["dW"], ws)
    torch.cuda.synchronize()
    fresh_status()
    return o


def _oracle_bwd(inp, Z, aq_val, r, s_a, s_dy, s_e, rows=None):
    rows = np.arange(inp["h"].shape[0]) if rows is None else rows
    return O.mlp_fp8_backward(f64(inp["h"])[rows], f64(inp["Xq"])[rows], inp["s_x"], f64(inp["Wq"]), inp["s_w"],
                              f64(inp["Wdq"]), inp["s_wd"], Z, aq_val, s_a, r, f64(inp["dY"])[rows], s_dy, s_e)


@pytest.mark.parametrize("M,H,F", [(384, 512, 768), (256, 256, 128)])
def test_fp8_backward_same_saved_tensors(C, M, H, F):
    inp = S.fp8_mlp_inputs(M, H, F, seed=1, with_grad=True)
    s_a = float(_oracle_fwd(inp, 1.0)["amax"]) / 448.0
    fo = _oracle_fwd(inp, s_a)
    # the saved tensors both sides get: Z as bf16, the a_q codes, r as fp32
    Zb = torch.from_numpy(fo["Z"]).to(torch.float32).to(BF)
    aq = torch.from_numpy(O.e4m3_encode(fo["aq_val"]))
    r32 = torch.from_numpy(fo["r"]).to(torch.float32)
    s_dy = float(np.max(np.abs(f64(inp["dY"])))) / 448.0
    pre = _oracle_bwd(inp, f64(Zb), fo["aq_val"], f64(r32), s_a, s_dy, 1.0)
    s_e = pre["amax_e"] / 448.0                           # delayed scaling from a prior pass
    ref = _oracle_bwd(inp, f64(Zb), fo["aq_val"], f64(r32), s_a, s_dy, s_e)
    got = _backward(C, inp, dev(Zb), dev(aq), dev(r32), s_a, s_dy, s_e)
    np.testing.assert_array_equal(got["dYq"].cpu().numpy(), _fp32_codes(f64(inp["dY"]), s_dy))
    assert float(got["amax_dy"].item()) == ref["amax_dy"]
    assert_e4m3_codes(got["eq"].cpu().numpy(), ref["e"] / s_e, "e codes")
    np.testing.assert_allclose(float(got["amax_e"].item()), ref["amax_e"], rtol=1e-3)
    assert_close(f64(got["c"]), ref["c"], TOL_FP8, "c")
    assert_close(f64(got["dh"]), ref["dh"], TOL_FP8, "dh")
    assert_close(f64(got["dW_d"]), ref["dW_d"], TOL_FP8, "dW_d")
    assert_close(f64(got["dW"]), ref["dW"], TOL_FP8, "dW")


def test_fp8_backward_empty_batch_zeroes_the_weight_gradients(C):
    H, F = 256, 128
    w = S.fp8_mlp_inputs(4, H, F, seed=2)
    e8 = torch.float8_e4m3fn
    inp = dict(h=torch.empty((0, H), dtype=BF), Xq=torch.empty((0, H), dtype=e8), Wq=w["Wq"], Wdq=w["Wdq"],
               dY=torch.empty((0, H), dtype=BF), s_x=w["s_x"], s_w=w["s_w"], s_wd=w["s_wd"])
    z = lambda *s, dt=BF: torch.empty(s, dtype=dt, device="cuda")
    o = _backward(C, inp, z(0, 2 * F), z(0, F, dt=U8), z(0, dt=torch.float32), 1.0, 1.0, 1.0)
    assert float(o["amax_dy"].item()) == 0.0 and float(o["amax_e"].item()) == 0.0
    assert torch.count_nonzero(o["dW_d"]) == 0 and torch.count_nonzero(o["dW"]) == 0


@pytest.mark.slow
def test_fp8_backward_full_size_end_to_end_sampled(C):
    """16384 tokens, H = 4096, F = 14336: GPU forward (saving Z) then GPU backward, against the
    oracle's forward + backward from the original inputs on sampled rows (row-local outputs)
    and sampled columns of the weight gradients (summed over all rows)."""
    M, H, F = 16384, 4096, 14336
    inp = S.fp8_mlp_inputs(M, H, F, seed=0, with_grad=True)
    rows = np.sort(np.concatenate([np.arange(64), np.random.default_rng(5).choice(np.arange(64, M), 64, False)]))
    s_a = 4.0 * float(_oracle_fwd(inp, 1.0, rows[:64])["amax"]) / 448.0
    fw = _forward(C, inp, s_a, True)
    s_dy = float(np.max(np.abs(f64(inp["dY"])))) / 448.0
    fo = _oracle_fwd(inp, s_a, rows)
    pre = _oracle_bwd(inp, fo["Z"], fo["aq_val"], fo["r"], s_a, s_dy, 1.0, rows)
    s_e = 4.0 * pre["amax_e"] / 448.0
    got = _backward(C, inp, fw["Z"], fw["aq"], fw["r"], s_a, s_dy, s_e)
    ref = _oracle_bwd(inp, fo["Z"], fo["aq_val"], fo["r"], s_a, s_dy, s_e, rows)
    np.testing.assert_array_equal(got["dYq"].cpu().numpy()[rows], _fp32_codes(f64(inp["dY"])[rows], s_dy))
    for k in ("c", "dh"):
        assert_close(f64(got[k])[rows], ref[k], TOL_FP8, k)
    # e codes: the GPU's e comes from its own bf16-stored Z, so a code may sit one step off
    # near a rounding midpoint.  Each code must be a rounding of x perturbed by 2% of |x|
    # plus 1% of the row's RMS (the absolute part covers elements near a zero of silu',
    # where a bf16 rounding of G moves e by a large fraction of itself but little in size)
    v = O.e4m3_decode(got["eq"].cpu().numpy()[rows])
    x = ref["e"] / s_e
    slack = 2e-2 * np.abs(x) + 1e-2 * np.sqrt(np.mean(x * x, axis=1, keepdims=True))
    lo, hi = O.e4m3_round(x - slack), O.e4m3_round(x + slack)
    assert np.all((v >= lo) & (v <= hi)), f"{int(np.sum(~((v >= lo) & (v <= hi))))} e codes outside the window"
    # bf16 storage moves e by ~0.1-0.4%, against an e4m3 step of 12.5%: a few percent of the
    # codes round the other way
    assert np.mean(v == O.e4m3_round(x)) >= 0.95
    # weight gradients on sampled columns, over all rows
    cols = np.sort(np.random.default_rng(6).choice(F, 32, replace=False))
    x_all = inp["s_x"] * f64(inp["Xq"])
    W = inp["s_w"] * f64(inp["Wq"])
    Wd = inp["s_wd"] * f64(inp["Wdq"])
    r_all = O.rms_scale(f64(inp["h"]), inp["eps"])
    G = r_all[:, None] * (x_all @ W[cols].T)
    U = r_all[:, None] * (x_all @ W[F + cols].T)
    a_q = O.e4m3_round(O.swiglu(G, U) / s_a)
    dYd = s_dy * O.e4m3_round(f64(inp["dY"]) / s_dy)
    assert_close(f64(got["dW_d"])[:, cols], dYd.T @ (s_a * a_q), TOL_FP8, "dW_d[:, cols]")
    dA = dYd @ Wd[:, cols]
    eg = r_all[:, None] * dA * U * O.silu_grad(G)
    eu = r_all[:, None] * dA * O.silu(G)
    q = lambda e: s_e * O.e4m3_round(e / s_e)
    # dW sums e4m3 codes of e, and a few percent of them round the other way on the GPU
    # because its e comes from the bf16-stored Z: bound the element-wise error by the same
    # storage model (Z rounded to bf16, tests/storage_sim), as for the bf16 product tensors
    Gs, Us = SIM.bf(G), SIM.bf(U)
    eg_s = r_all[:, None] * dA * Us * O.silu_grad(Gs)
    eu_s = r_all[:, None] * dA * O.silu(Gs)
    for name, idx, e_ref, e_sim in (("gate", cols, eg, eg_s), ("up", F + cols, eu, eu_s)):
        ref_dW, sim_dW = q(e_ref).T @ x_all, q(e_sim).T @ x_all
        got_dW = f64(got["dW"])[idx]
        assert normwise(got_dW, ref_dW) <= TOL_FP8, name
        el, el_sim = O.max_rel_err(got_dW, ref_dW), O.max_rel_err(sim_dW, ref_dW)
        assert el <= max(TOL_FP8, 1.5 * el_sim), f"dW[{name} cols]: {el:.3e} (storage model {el_sim:.3e})"
