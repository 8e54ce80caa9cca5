"""GPU parity of each compiled epilogue program against the fp64 oracle, through the C ABI.

Sizes span several 128 x 256 tiles and leave ragged tails in M, N and K.  Inputs are
seeded; the oracle sees the exact values the GPU sees (bf16 / fp32 / e4m3 widened to
float64).  Tolerance: max relative error (RMS floor) 2e-2 for bf16 and tf32 outputs."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_helpers import TOL_BF16, TOL_FP8, assert_close, assert_e4m3_codes, dev, f64, fresh_status, seeded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


BF = torch.bfloat16


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 288, 200), (513, 768, 1000),
                                   (1, 32, 8), (7, 64, 16)])   # degenerate: one row, the narrowest N, K of one TMA row
def test_plain_bf16(C, M, N, K):
    A = seeded((M, K), 1, dtype=BF)
    W = seeded((N, K), 2, std=0.05, dtype=BF)
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [], out)
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), O.linear(f64(A), f64(W)), TOL_BF16, "A W^T")


def test_plain_f32_out_and_tensor_scale(C):
    M, N, K = 200, 512, 136
    A = seeded((M, K), 3, dtype=BF)
    W = seeded((N, K), 4, std=0.05, dtype=BF)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_TENSOR_SCALE], out, tensor_scale=0.5)
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), 0.5 * O.linear(f64(A), f64(W)), 1e-5, "0.5 A W^T (fp32 out)")


def test_residual_and_partial_sumsq(C):
    M, N, K = 300, 512, 256
    A = seeded((M, K), 5, dtype=BF)
    W = seeded((N, K), 6, std=0.05, dtype=BF)
    R = seeded((M, N), 7, dtype=BF)
    out = torch.empty((M, N), dtype=BF, device="cuda")
    P = torch.full((2, M + 4), -1.0, dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL], out, residual=dev(R),
                         row_partials=P)
    torch.cuda.synchronize()
    fresh_status()
    h = O.linear(f64(A), f64(W)) + f64(R)
    assert_close(f64(out), h, TOL_BF16, "A W^T + R")
    Pg = f64(P)
    assert_close(Pg[:, :M], O.partial_sumsq(h, 256), TOL_BF16, "partial sums of squares")
    assert np.all(Pg[:, M:] == -1.0), "wrote past M in the partials"


def test_rowscale(C):
    M, N, K = 256, 256, 512
    A = seeded((M, K), 8, dtype=BF)
    W = seeded((N, K), 9, std=0.05, dtype=BF)
    r = seeded((M,), 10, std=0.2, mean=1.0)
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_ROW_SCALE], out, row_scale=dev(r))
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), f64(r)[:, None] * O.linear(f64(A), f64(W)), TOL_BF16, "r * A W^T")


@pytest.mark.parametrize("save_z", [False, True])
def test_rowscale_swiglu(C, save_z):
    M, F, K = 300, 384, 256
    A = seeded((M, K), 11, dtype=BF)
    W = seeded((2 * F, K), 12, std=0.08, dtype=BF)
    r = seeded((M,), 13, std=0.2, mean=1.0)
    out = torch.empty((M, F), dtype=BF, device="cuda")
    Z = torch.empty((M, 2 * F), dtype=BF, device="cuda") if save_z else None
    ops = [C.OP_ROW_SCALE, C.OP_STORE_AUX, C.OP_SWIGLU] if save_z else [C.OP_ROW_SCALE, C.OP_SWIGLU]
    C.coda_gemm_epilogue(dev(A), dev(W), ops, out, row_scale=dev(r), store_aux=Z)
    torch.cuda.synchronize()
    fresh_status()
    Zr = f64(r)[:, None] * O.linear(f64(A), f64(W))
    assert_close(f64(out), O.swiglu(Zr[:, :F], Zr[:, F:]), TOL_BF16, "silu(G) U")
    if save_z:
        assert_close(f64(Z), Zr, TOL_BF16, "saved Z")


def test_rowscale_rope(C):
    M, N, K, hd, seq = 256, 768, 256, 64, 100
    A = seeded((M, K), 14, dtype=BF)
    W = seeded((N, K), 15, std=0.05, dtype=BF)
    r = seeded((M,), 16, std=0.2, mean=1.0)
    cos = torch.empty((seq, hd // 2), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, 500000.0, cos, sin)
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_ROW_SCALE, C.OP_ROPE], out, row_scale=dev(r), rope_cos=cos,
                         rope_sin=sin, rope_seq_len=seq, rope_head_dim=hd, rope_ncols=640)
    torch.cuda.synchronize()
    fresh_status()
    Z = f64(r)[:, None] * O.linear(f64(A), f64(W))
    ref = O.rope_rotate(Z, np.arange(M) % seq, 640, hd, 500000.0)
    assert_close(f64(out), ref, TOL_BF16, "rope(r A W^T)")


def test_rope_table(C):
    seq, hd = 1024, 64
    cos = torch.empty((seq, hd // 2), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, 500000.0, cos, sin)
    torch.cuda.synchronize()
    phi = np.arange(seq)[:, None] * O.rope_inv_freq(hd, 500000.0)[None, :]
    np.testing.assert_allclose(f64(cos), np.cos(phi), atol=1e-7)
    np.testing.assert_allclose(f64(sin), np.sin(phi), atol=1e-7)


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (384, 256, 520)])
def test_mn_major_operands(C, M, N, K):
    # dW-type: A = X^T, B = Y^T views of row-major [K, M] / [K, N] activations, fp32 out
    X = seeded((K, M), 17, dtype=BF)
    Y = seeded((K, N), 18, std=0.1, dtype=BF)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(X).t(), dev(Y).t(), [], out)
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), f64(X).T @ f64(Y), 1e-5, "X^T Y")
    # dX-type: B = W^T view of a row-major [K, N] weight, bf16 out
    A = seeded((M, K), 19, dtype=BF)
    Wt = seeded((K, N), 20, std=0.05, dtype=BF)
    out2 = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(Wt).t(), [], out2)
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out2), f64(A) @ f64(Wt), TOL_BF16, "A W (W stored [K, N])")


def test_colscale_mn_major(C):
    M, N, K = 512, 256, 300
    X = seeded((K, M), 21, dtype=BF)
    Y = seeded((K, N), 22, dtype=BF)
    g = seeded((N,), 23, std=0.1, mean=1.0)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(X).t(), dev(Y).t(), [C.OP_COL_SCALE], out, col_scale=dev(g))
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), (f64(X).T @ f64(Y)) * f64(g)[None, :], 1e-5, "(X^T Y) g")


@pytest.mark.parametrize("M,F,ts", [(300, 512, None), (300, 288, 0.5)])
def test_swiglu_backward_epilogue(C, M, F, ts):
    """F = 288: the second 256-column tile has one live 32-column chunk, so the gate and up
    blocks of Z and e (moved as one 3-D box) are clipped at F in both halves."""
    H = 256
    dY = seeded((M, H), 24, dtype=BF)
    Wd = seeded((H, F), 25, std=0.05, dtype=BF)       # stored [H, F]; the GEMM reads W_d^T
    Z = seeded((M, 2 * F), 26, dtype=BF)
    r = seeded((M,), 27, std=0.2, mean=1.0)
    e = torch.full((M, 2 * F), float("nan"), dtype=BF, device="cuda")
    nt = (F + 255) // 256
    S = torch.empty((nt, M), dtype=torch.float32, device="cuda")
    ops = [C.OP_SWIGLU_BWD, C.OP_ROW_SCALE, C.OP_ROW_DOT_PARTIAL]
    if ts is not None:
        ops = [C.OP_TENSOR_SCALE] + ops
    C.coda_gemm_epilogue(dev(dY), dev(Wd).t(), ops, e, aux_in=dev(Z), row_scale=dev(r), row_partials=S,
                         tensor_scale=ts if ts is not None else 1.0)
    torch.cuda.synchronize()
    fresh_status()
    dA = (ts if ts is not None else 1.0) * (f64(dY) @ f64(Wd))
    G, U = f64(Z)[:, :F], f64(Z)[:, F:]
    ref = f64(r)[:, None] * np.hstack([dA * U * O.silu_grad(G), dA * O.silu(G)])
    assert_close(f64(e), ref, TOL_BF16, "e")
    s_ref = np.stack([np.sum((ref * f64(Z))[:, np.r_[t * 256:min((t + 1) * 256, F), F + t * 256:F + min((t + 1) * 256,
                                                                                                    F)]], axis=1)
                      for t in range(nt)])
    assert_close(f64(S), s_ref, TOL_BF16, "row partials of e . Z")


def test_rmsnorm_backward_without_gain_and_scaled(C):
    """The combine with a tensor scale and no gain (g = 1, no column partials), the form the
    FP8 backward uses, at a ragged width (H = 288)."""
    M, H, K = 300, 288, 384
    E = seeded((M, K), 34, dtype=BF)
    W = seeded((K, H), 35, std=0.05, dtype=BF)
    h = seeded((M, H), 36, dtype=BF)
    dY = seeded((M, H), 37, dtype=BF)
    c = seeded((M,), 38, std=0.1)
    out = torch.empty((M, H), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(dev(E), dev(W).t(), [C.OP_TENSOR_SCALE, C.OP_RMSBWD_COMBINE], out, aux_in=dev(h),
                         aux_in2=dev(dY), row_coef=dev(c), tensor_scale=0.25)
    torch.cuda.synchronize()
    fresh_status()
    ref = 0.25 * (f64(E) @ f64(W)) - f64(c)[:, None] * f64(h) + f64(dY)
    assert_close(f64(out), ref, TOL_BF16, "s t - c h + dY")


def test_rmsnorm_backward_epilogue(C):
    M, H, K = 300, 512, 384
    E = seeded((M, K), 28, dtype=BF)
    Wgu = seeded((K, H), 29, std=0.05, dtype=BF)      # stored [2F, H]; the GEMM reads W_gu^T
    h = seeded((M, H), 30, dtype=BF)
    dY = seeded((M, H), 31, dtype=BF)
    g = seeded((H,), 32, std=0.1, mean=1.0)
    c = seeded((M,), 33, std=0.1)
    out = torch.empty((M, H), dtype=BF, device="cuda")
    nblk = (M + 31) // 32
    Dg = torch.empty((nblk, H), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(E), dev(Wgu).t(), [C.OP_RMSBWD_COMBINE, C.OP_COL_DOT_PARTIAL], out, aux_in=dev(h),
                         aux_in2=dev(dY), col_scale=dev(g), row_coef=dev(c), col_partials=Dg)
    dg = torch.empty((H,), dtype=torch.float32, device="cuda")
    C.coda_col_reduce(Dg, dg)
    torch.cuda.synchronize()
    fresh_status()
    t = f64(E) @ f64(Wgu)
    ref = f64(g)[None, :] * t - f64(c)[:, None] * f64(h) + f64(dY)
    assert_close(f64(out), ref, TOL_BF16, "g t - c h + dY")
    assert_close(f64(dg), np.sum(f64(h) * t, axis=0), 1e-4, "column sums of h t")


def test_tf32_residual_and_rowscale(C):
    M, N, K = 200, 256, 256
    A = seeded((M, K), 34)
    W = seeded((N, K), 35, std=1 / 16)
    R = seeded((M, N), 36)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    P = torch.empty((1, M), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL], out, residual=dev(R),
                         row_partials=P)
    torch.cuda.synchronize()
    fresh_status()
    h = O.linear(f64(A), f64(W)) + f64(R)
    assert_close(f64(out), h, TOL_BF16, "tf32 A W^T + R")
    r = seeded((M,), 37, std=0.2, mean=1.0)
    out2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(A), dev(W), [C.OP_ROW_SCALE], out2, row_scale=dev(r))
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out2), f64(r)[:, None] * O.linear(f64(A), f64(W)), TOL_BF16, "tf32 r A W^T")


def _e4m3(x, scale):
    return (x / scale).clamp(-448, 448).to(torch.float8_e4m3fn)


def test_fp8_swiglu_requant_and_residual(C):
    M, F, K = 300, 256, 512
    x = seeded((M, K), 38)
    w = seeded((2 * F, K), 39, std=0.05)
    sx, sw = float(x.abs().max()) / 448, float(w.abs().max()) / 448
    Xq, Wq = _e4m3(x, sx), _e4m3(w, sw)
    r = seeded((M,), 40, std=0.2, mean=1.0)
    Zr = f64(r)[:, None] * (sx * f64(Xq)) @ (sw * f64(Wq)).T
    a_ref = O.swiglu(Zr[:, :F], Zr[:, F:])
    sa = float(np.abs(a_ref).max()) / 448
    aq = torch.empty((M, F), dtype=torch.uint8, device="cuda")
    amax = torch.zeros((1,), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(dev(Xq), dev(Wq), [C.OP_TENSOR_SCALE, C.OP_ROW_SCALE, C.OP_SWIGLU, C.OP_AMAX], aq,
                         tensor_scale=sx * sw, row_scale=dev(r), out_scale=1.0 / sa, amax=amax)
    torch.cuda.synchronize()
    fresh_status()
    codes = aq.cpu().numpy()
    assert_e4m3_codes(codes, a_ref / sa, "a_q codes")
    got = sa * O.e4m3_decode(codes)
    assert_close(got, a_ref, TOL_FP8 * 2.2, "dequantised a_q (one e4m3 rounding)")
    np.testing.assert_allclose(float(amax.item()), np.abs(a_ref).max(), rtol=1e-2)
    # down GEMM in e4m3 with residual and partials
    H = 256
    wd = seeded((H, F), 41, std=0.05)
    swd = float(wd.abs().max()) / 448
    Wdq = _e4m3(wd, swd)
    h = seeded((M, H), 42, dtype=BF)
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((1, M), dtype=torch.float32, device="cuda")
    C.coda_gemm_epilogue(aq.view(torch.float8_e4m3fn), dev(Wdq), [C.OP_TENSOR_SCALE, C.OP_ADD_SIDE,
                         C.OP_ROW_SUMSQ_PARTIAL], Y, tensor_scale=sa * swd, residual=dev(h), row_partials=P)
    torch.cuda.synchronize()
    fresh_status()
    Yref = got @ (swd * f64(Wdq)).T + f64(h)
    assert_close(f64(Y), Yref, TOL_BF16, "fp8 down + residual")
    assert_close(f64(P), O.partial_sumsq(Yref, 256), TOL_BF16, "fp8 partials")


def test_partial_reduce_and_row_rms(C):
    M, d = 1000, 2048
    X = seeded((M, d), 43, std=2.0, dtype=BF)
    r = torch.empty((M,), dtype=torch.float32, device="cuda")
    C.coda_row_rms(dev(X), 1e-6, r)
    P = torch.tensor(O.partial_sumsq(f64(X), 256), dtype=torch.float32, device="cuda")
    r2 = torch.empty_like(r)
    C.coda_rms_partial_reduce(P, M, d, 1e-6, r2)
    torch.cuda.synchronize()
    ref = O.rms_scale(f64(X), 1e-6)
    assert_close(f64(r), ref, 1e-5, "row rms")
    assert_close(f64(r2), ref, 1e-5, "partial reduce")


@pytest.mark.parametrize("nparts", [1, 3, 8, 37, 501])
def test_partial_reduce_many_parts(C, nparts):
    """The reduce splits a row's parts over eight warps and merges them in a fixed order: every
    part count (fewer than the warps, not a multiple of them, the LM head's 501) against the
    plain sums, with a ragged number of rows, in both modes, and bit-identical run to run."""
    M, d = 1000, 2048
    g = np.random.default_rng(nparts)
    Pn = g.uniform(0.0, 4.0, size=(nparts, M))
    P = torch.tensor(Pn, dtype=torch.float32, device="cuda")
    r1, r2 = torch.empty((M,), device="cuda"), torch.empty((M,), device="cuda")
    C.coda_rms_partial_reduce(P, M, d, 1e-6, r1)
    C.coda_rms_partial_reduce(P, M, d, 1e-6, r2)
    rs = torch.tensor(g.uniform(0.5, 1.5, size=M), dtype=torch.float32, device="cuda")
    c = torch.empty((M,), device="cuda")
    C.coda_rms_partial_reduce(P, M, d, 0.0, c, mode=C.REDUCE_SCALE_SUM, rowscale=rs)
    torch.cuda.synchronize()
    fresh_status()
    assert torch.equal(r1, r2), "not reproducible"
    tot = np.sum(f64(P), axis=0)
    assert_close(f64(r1), 1.0 / np.sqrt(tot / d + 1e-6), 1e-5, f"r from {nparts} parts")
    assert_close(f64(c), f64(rs) * tot / d, 1e-5, f"c = r s / d from {nparts} parts")


@pytest.mark.parametrize("nparts", [4, 37, 501])
def test_xent_combine_many_tiles(C, nparts):
    """The cross-entropy combine folds the tile states into eight running (max, scaled sum)
    pairs and merges them in order: against the oracle's combine for several tile counts, a
    ragged number of rows, a tile state with no column (max -inf, sum 0) that must be ignored,
    and bit-identical run to run."""
    M, V = 1000, 256 * nparts
    g = np.random.default_rng(100 + nparts)
    m = g.normal(0.0, 3.0, size=(nparts, M))
    s = g.uniform(1.0, 256.0, size=(nparts, M))
    if nparts > 1:
        m[nparts // 2, :7] = -np.inf   # rows 0..6: one tile without columns
        s[nparts // 2, :7] = 0.0
    Pm = torch.tensor(m, dtype=torch.float32, device="cuda")
    Ps = torch.tensor(s, dtype=torch.float32, device="cuda")
    T = torch.tensor(g.normal(size=M), dtype=torch.float32, device="cuda")
    tg = torch.tensor(g.integers(0, V, size=M), dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        lse, loss, mean = (torch.empty((n,), device="cuda") for n in (M, M, 1))
        C.coda_xent_combine(Pm, Ps, T, tg, V, lse, loss, mean)
        outs.append((lse, loss, mean))
    torch.cuda.synchronize()
    fresh_status()
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1])), "not reproducible"
    keep = np.isfinite(m)
    ref = O.xent_combine(np.where(keep, m, -1e300), np.where(keep, s, 0.0))
    assert_close(f64(outs[0][0]), ref, 1e-6, f"lse from {nparts} tiles")
    assert_close(f64(outs[0][1]), ref - f64(T), 1e-5, "loss")


def test_fold_gain(C):
    N, K = 300, 512
    W = seeded((N, K), 44, std=0.05, dtype=BF)
    g = seeded((K,), 45, std=0.1, mean=1.0)
    out = torch.empty((N, K), dtype=BF, device="cuda")
    C.coda_fold_gain(dev(W), dev(g), out)
    torch.cuda.synchronize()
    assert_close(f64(out), O.fold_gain(f64(W), f64(g)), 4e-3, "W diag(g)")


def test_empty_m_is_noop(C):
    A = torch.empty((0, 64), dtype=BF, device="cuda")
    W = seeded((256, 64), 46, dtype=BF).cuda()
    out = torch.empty((0, 256), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(A, W, [], out)
    torch.cuda.synchronize()
    fresh_status()


def test_rejections_launch_nothing(C):
    A = seeded((128, 64), 47, dtype=BF).cuda()
    W = seeded((256, 64), 48, dtype=BF).cuda()
    out = torch.empty((128, 256), dtype=BF, device="cuda")
    with pytest.raises(C.CodaError) as ei:
        C.coda_gemm_epilogue(A, W, [C.OP_ROW_SUMSQ_PARTIAL, C.OP_ADD_SIDE], out)
    assert ei.value.status == C.ERR_UNSUPPORTED_PROGRAM
    with pytest.raises(C.CodaError) as ei:
        C.coda_gemm_epilogue(A, W[:, :32], [], out)
    assert ei.value.status == C.ERR_SHAPE
    with pytest.raises(C.CodaError) as ei:
        C.coda_gemm_epilogue(A, W, [C.OP_ROW_SCALE], out)
    assert ei.value.status == C.ERR_NULL
    bad = torch.empty((128, 64 + 4), dtype=BF, device="cuda")[:, :60]
    with pytest.raises(C.CodaError) as ei:
        C.coda_gemm_epilogue(bad, W[:, :60], [], out)
    assert ei.value.status == C.ERR_ALIGN
    fresh_status()


@pytest.mark.parametrize("M,N,K,colscale", [(256, 512, 16384, False), (384, 256, 9000, True)])
def test_split_k_reduce_add(C, M, N, K, colscale):
    # few output tiles and a long K: the library splits K and reduce-adds the fp32 partials
    X = seeded((K, M), 80, dtype=BF)
    Y = seeded((K, N), 81, std=0.1, dtype=BF)
    g = seeded((N,), 82, std=0.1, mean=1.0)
    out = torch.full((M, N), 123.0, device="cuda")       # must be overwritten, not added to
    ops = [C.OP_COL_SCALE] if colscale else []
    C.coda_gemm_epilogue(dev(X).t(), dev(Y).t(), ops, out, col_scale=dev(g) if colscale else None)
    torch.cuda.synchronize()
    fresh_status()
    ref = f64(X).T @ f64(Y)
    if colscale:
        ref = ref * f64(g)[None, :]
    assert_close(f64(out), ref, 1e-5, "split-K X^T Y")


def test_padded_leading_dimensions(C):
    """Operands, residual and output as column slices of wider buffers (ld > cols): the tensor
    maps take their strides from ld, and nothing outside the slices is written."""
    M, N, K = 300, 256, 200
    A_full = seeded((M, K + 56), 80, dtype=BF)                 # ld 256 for a [300, 200] A
    W_full = seeded((N, K + 24), 81, std=0.05, dtype=BF)        # ld 224 for a [256, 200] W
    R_full = seeded((M, N + 64), 82, dtype=BF)
    A, W, R = dev(A_full)[:, :K], dev(W_full)[:, :K], dev(R_full)[:, 8:8 + N]
    out_full = torch.full((M, N + 32), 7.0, dtype=BF, device="cuda")
    out = out_full[:, 16:16 + N]
    C.coda_gemm_epilogue(A, W, [C.OP_ADD_SIDE], out, residual=R)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(f64(A_full)[:, :K], f64(W_full)[:, :K]) + f64(R_full)[:, 8:8 + N]
    assert_close(f64(out), ref, TOL_BF16, "A W^T + R through padded views")
    got = f64(out_full)
    assert np.all(got[:, :16] == 7.0) and np.all(got[:, 16 + N:] == 7.0), "wrote outside the output slice"


def test_nvfp4_padded_codes(C):
    """NVFP4 operands whose code rows are wider than K / 2 bytes (ld > cols)."""
    from tests import nvfp4_layout as L
    M, N, K = 256, 256, 512
    g = torch.Generator().manual_seed(83)
    xa = f64(torch.randn((M, K), generator=g).to(BF))
    xb = f64((torch.randn((N, K), generator=g) * 0.05).to(BF))
    sc = lambda x: float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    A, qa, sfa = L.oracle_nvfp4(xa, sc(xa))
    B, qb, sfb = L.oracle_nvfp4(xb, sc(xb))
    pad = torch.zeros((M, K // 2 + 48), dtype=torch.uint8, device="cuda")
    pad[:, :K // 2] = A.codes
    A.codes = pad[:, :K // 2]                                   # rows K/2 + 48 bytes apart
    out = torch.empty((M, N), device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out, tensor_scale=A.s * B.s)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s))
    assert_close(f64(out), ref, 1e-3, "NVFP4 GEMM with padded code rows")
