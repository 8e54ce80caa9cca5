"""Pins for the fp64 oracle: closed forms, invariants, library special cases, brute force
and finite differences.  None of them re-types the oracle's own formula: each checks the
oracle against something that fixes the answer independently, chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one of them.

Sources: [Ecosistema] "CODA: Nuevo kernel GPU reduce costos de entrenamiento IA",
section "¿Qué es GEMM-epilogue…?" (GEMM C = alpha*A*B + beta*C); [KuCoin] "CODA: new
research optimizes Transformer training with GEMM-epilogue programming", sections
"El epílogo esconde un tesoro" (deferred r, partial RMS, backward inherits the
structure) and "Cinco bloques y un lenguaje LEGO" (the primitive kinds)."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------------------ GEMM
def test_gemm_brute_force_triple_loop():
    A = RNG.normal(size=(5, 7))
    B = RNG.normal(size=(7, 3))
    C = RNG.normal(size=(5, 3))
    ref = np.zeros((5, 3))
    for i, j in itertools.product(range(5), range(3)):
        ref[i, j] = 0.5 * sum(A[i, k] * B[k, j] for k in range(7)) + 2.0 * C[i, j]
    np.testing.assert_allclose(O.gemm_general(A, B, alpha=0.5, C=C, beta=2.0), ref, rtol=1e-13, atol=1e-13)


def test_linear_identity_and_ones():
    X = RNG.normal(size=(6, 4))
    np.testing.assert_array_equal(O.linear(X, np.eye(4)), X)
    ones = np.ones((1, 4))  # one output column = row sums
    np.testing.assert_allclose(O.linear(X, ones)[:, 0], X.sum(axis=1), rtol=1e-14)


def test_linear_uses_out_in_layout():
    # W stored [out, in]: a weight with distinct out/in sizes only multiplies one way.
    X = RNG.normal(size=(3, 5))
    W = RNG.normal(size=(2, 5))
    Y = O.linear(X, W)
    assert Y.shape == (3, 2)
    np.testing.assert_allclose(Y[1, 0], np.dot(X[1], W[0]), rtol=1e-14)


# --------------------------------------------------------------------------- RMSNorm
def test_rms_constant_row():
    c, d, eps = 1.7, 64, 1e-6
    h = np.full((2, d), c)
    np.testing.assert_allclose(O.rms_scale(h, eps), 1.0 / math.sqrt(c * c + eps), rtol=1e-15)


def test_rms_single_nonzero():
    d, a, eps = 32, -3.0, 0.0
    h = np.zeros((1, d))
    h[0, 5] = a
    # rms = |a| / sqrt(d)
    np.testing.assert_allclose(O.rms_scale(h, eps)[0], math.sqrt(d) / abs(a), rtol=1e-15)


def test_rms_eps_only_row():
    np.testing.assert_allclose(O.rms_scale(np.zeros((1, 8)), 0.25), 2.0, rtol=1e-15)


def test_rmsnorm_output_has_unit_rms():
    h = RNG.normal(size=(4, 128)) * 5.0
    y = O.rmsnorm(h, np.ones(128), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)


def test_rmsnorm_gain_is_per_column():
    h = RNG.normal(size=(3, 16))
    g = RNG.normal(size=16)
    y1 = O.rmsnorm(h, np.ones(16), 1e-6)
    y2 = O.rmsnorm(h, g, 1e-6)
    np.testing.assert_allclose(y2, y1 * g[None, :], rtol=1e-14)


@pytest.mark.parametrize("bn", [32, 64, 256, 2048, 100])
def test_partials_sum_to_row_sumsq(bn):
    h = RNG.normal(size=(9, 2048))
    P = O.partial_sumsq(h, bn)
    assert P.shape == ((2048 + bn - 1) // bn, 9)
    np.testing.assert_allclose(P.sum(axis=0), (h ** 2).sum(axis=1), rtol=1e-13)
    np.testing.assert_allclose(O.rms_scale_from_partials(P, 2048, 1e-6), O.rms_scale(h, 1e-6), rtol=1e-13)


def test_row_scale_commutes_with_gemm():
    # diag(r)(X W) = (diag(r) X) W: the algebraic fact the reparameterisation rests on.
    X = RNG.normal(size=(7, 11))
    W = RNG.normal(size=(11, 5))
    r = RNG.uniform(0.1, 3.0, size=7)
    lhs = r[:, None] * O.gemm_general(X, W)
    rhs = O.gemm_general(r[:, None] * X, W)
    assert np.max(np.abs(lhs - rhs) / np.maximum(np.abs(rhs), 1e-300)) <= 1e-12


def test_fold_gain_equals_scaling_input():
    h = RNG.normal(size=(5, 8))
    W = RNG.normal(size=(6, 8))
    g = RNG.normal(size=8)
    np.testing.assert_allclose(O.linear(h, O.fold_gain(W, g)), O.linear(h * g[None, :], W), rtol=1e-12)


def _block(M=5, d=8, F=4, seed=0):
    rng = np.random.default_rng(seed)
    return dict(
        O=rng.normal(size=(M, d)), R=rng.normal(size=(M, d)),
        W_o=rng.normal(size=(d, d)) / 3, g=1 + 0.1 * rng.normal(size=d),
        W_gu=rng.normal(size=(2 * F, d)) / 3, W_d=rng.normal(size=(d, F)) / 3, eps=1e-6,
    )


def test_deferred_r_equals_naive():
    b = _block(M=16, d=64, F=32)
    naive = O.block_forward(b["O"], b["R"], b["W_o"], b["g"], b["W_gu"], b["W_d"], b["eps"])
    for bn in (16, 32, 64):
        fused = O.block_forward_deferred(b["O"], b["R"], b["W_o"], b["g"], b["W_gu"], b["W_d"], b["eps"], bn)
        for k in ("h", "r", "Z", "a", "Y"):
            ref = naive[k]
            assert np.max(np.abs(fused[k] - ref)) <= 1e-12 * np.max(np.abs(ref)), k


# --------------------------------------------------------------------------- SwiGLU
def test_sigmoid_closed_forms_and_symmetry():
    assert O.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(O.sigmoid(math.log(3.0)), 0.75, rtol=1e-15)     # 1 / (1 + 1/3)
    x = np.linspace(-30.0, 30.0, 121)
    np.testing.assert_allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    # the derivative is sigma (1 - sigma): central differences, whose rounding error is at most
    # eps / h = 2.2e-11 and whose truncation error is below h^2 / 6 * max |sigma'''| < 2e-12
    h = 1e-5
    np.testing.assert_allclose((O.sigmoid(x + h) - O.sigmoid(x - h)) / (2 * h),
                               O.sigmoid(x) * (1 - O.sigmoid(x)), rtol=1e-6, atol=5e-11)


def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    np.testing.assert_allclose(O.silu(40.0), 40.0, rtol=1e-15)
    assert abs(O.silu(-40.0)) < 1e-15
    np.testing.assert_allclose(O.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(O.silu_grad(0.0), 0.5, rtol=1e-15)


def test_silu_grad_finite_difference():
    x = np.linspace(-6, 6, 41)
    h = 1e-6
    fd = (O.silu(x + h) - O.silu(x - h)) / (2 * h)
    np.testing.assert_allclose(O.silu_grad(x), fd, rtol=1e-7, atol=1e-9)


def test_swiglu_gate_and_up_roles():
    G = np.array([[0.0, 2.0]])
    U = np.array([[5.0, 3.0]])
    np.testing.assert_allclose(O.swiglu(G, U), [[0.0, 3.0 * 2.0 / (1 + math.exp(-2.0))]], rtol=1e-15)


# ----------------------------------------------------------------------------- RoPE
def _rope_setup(M=6, head_dim=8, heads=3):
    Z = RNG.normal(size=(M, head_dim * heads))
    return Z, head_dim, heads


def test_rope_position_zero_is_identity():
    Z, hd, nh = _rope_setup()
    out = O.rope_rotate(Z, np.zeros(Z.shape[0]), hd * nh, hd, 10000.0)
    np.testing.assert_array_equal(out, Z)


def test_rope_preserves_pair_norms_and_skips_unrotated_columns():
    Z, hd, nh = _rope_setup()
    pos = np.arange(Z.shape[0]) * 7
    out = O.rope_rotate(Z, pos, 2 * hd, hd, 500000.0)
    n_in = Z[:, :2 * hd:2] ** 2 + Z[:, 1:2 * hd:2] ** 2
    n_out = out[:, :2 * hd:2] ** 2 + out[:, 1:2 * hd:2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13)
    np.testing.assert_array_equal(out[:, 2 * hd:], Z[:, 2 * hd:])


def test_rope_closed_form_first_pair():
    # pair p = 0 has theta_0 = 1: a rotation by `pos` radians of (x0, x1)
    Z = np.zeros((1, 4))
    Z[0, 0], Z[0, 1] = 1.0, 0.0
    out = O.rope_rotate(Z, np.array([2.0]), 4, 4, 10000.0)
    np.testing.assert_allclose(out[0, :2], [math.cos(2.0), math.sin(2.0)], rtol=1e-15)
    # pair p = 1 of a head_dim-4 head: theta_1 = base^(-1/2)
    Z = np.zeros((1, 4))
    Z[0, 2], Z[0, 3] = 0.0, 1.0
    out = O.rope_rotate(Z, np.array([3.0]), 4, 4, 10000.0)
    phi = 3.0 / 100.0
    np.testing.assert_allclose(out[0, 2:], [-math.sin(phi), math.cos(phi)], rtol=1e-14)


def test_rope_relative_position_property():
    # <RoPE(q, m), RoPE(k, n)> depends only on m - n
    hd = 16
    q = RNG.normal(size=(1, hd))
    k = RNG.normal(size=(1, hd))

    def dot(m, n):
        qm = O.rope_rotate(q, np.array([m]), hd, hd, 500000.0)
        kn = O.rope_rotate(k, np.array([n]), hd, hd, 500000.0)
        return float(np.sum(qm * kn))

    np.testing.assert_allclose(dot(10, 3), dot(107, 100), rtol=1e-12)
    np.testing.assert_allclose(dot(0, 5), dot(1000, 1005), rtol=1e-11)


def test_rope_commutes_with_row_scale():
    Z, hd, nh = _rope_setup()
    r = RNG.uniform(0.5, 2, size=Z.shape[0])
    pos = np.arange(Z.shape[0]) + 3
    np.testing.assert_allclose(O.rope_rotate(r[:, None] * Z, pos, hd * nh, hd, 1e4),
                               r[:, None] * O.rope_rotate(Z, pos, hd * nh, hd, 1e4), rtol=1e-13)


# ------------------------------------------------------------------------------ FP8
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    np.testing.assert_array_equal(np.isnan(mine), nan)
    np.testing.assert_array_equal(mine[~nan], lib[~nan])
    assert np.nanmax(mine) == 448.0 and mine[1] == 2.0 ** -9


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    np.testing.assert_array_equal(O.e4m3_encode(vals), codes)
    np.testing.assert_array_equal(O.e4m3_round(vals), vals)


def test_e4m3_ties_to_even_and_saturation():
    # between 1.0 (mantissa 0) and 1.125 (mantissa 1) the tie goes to the even mantissa
    assert O.e4m3_round(1.0625) == 1.0
    assert O.e4m3_round(1.1875) == 1.25          # tie between m=1 and m=2 -> even m=2
    assert O.e4m3_round(-1.0625) == -1.0
    assert O.e4m3_round(1e6) == 448.0 and O.e4m3_round(-1e6) == -448.0
    assert O.e4m3_round(2.0 ** -10) == 0.0       # half of the smallest subnormal -> even (0)
    assert O.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8


def test_e4m3_round_matches_torch_cast_in_range():
    x = RNG.normal(size=20000) * 60.0
    x = np.clip(x, -448, 448)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_round(x), lib)


# ------------------------------------------------------------------------- backward
def _loss_grads_fd(b, dY, eps_fd=1e-6):
    names = ["O", "R", "W_o", "g", "W_gu", "W_d"]

    def loss(args):
        f = O.block_forward(*[args[n] for n in names], b["eps"])
        return float(np.sum(f["Y"] * dY))

    grads = {}
    for n in names:
        base = {k: b[k].copy() for k in names}
        gmat = np.zeros_like(b[n])
        for ix in np.ndindex(b[n].shape):
            p = {k: v.copy() for k, v in base.items()}
            m = {k: v.copy() for k, v in base.items()}
            p[n][ix] += eps_fd
            m[n][ix] -= eps_fd
            gmat[ix] = (loss(p) - loss(m)) / (2 * eps_fd)
        grads[n] = gmat
    return grads


def test_backward_matches_finite_differences():
    b = _block()
    dY = np.random.default_rng(7).normal(size=(5, 8))
    fwd = O.block_forward(b["O"], b["R"], b["W_o"], b["g"], b["W_gu"], b["W_d"], b["eps"])
    an = O.block_backward(fwd, b["O"], b["W_o"], b["g"], b["W_gu"], b["W_d"], dY)
    fd = _loss_grads_fd(b, dY)
    pairs = dict(O="dO", R="dR", W_o="dW_o", g="dg", W_gu="dW_gu", W_d="dW_d")
    for n, k in pairs.items():
        err = np.max(np.abs(an[k] - fd[n])) / np.max(np.abs(fd[n]))
        assert err <= 1e-6, (k, err)


def test_fused_backward_equals_plain_chain_rule():
    b = _block(M=12, d=32, F=16, seed=3)
    dY = np.random.default_rng(8).normal(size=(12, 32))
    fwd = O.block_forward(b["O"], b["R"], b["W_o"], b["g"], b["W_gu"], b["W_d"], b["eps"])
    plain = O.block_backward(fwd, b["O"], b["W_o"], b["g"], b["W_gu"], b["W_d"], dY)
    fused = O.block_backward_fused(fwd, b["O"], b["W_o"], b["g"], b["W_gu"], b["W_d"], dY)
    for k in ("dh", "dR", "dO", "dW_o", "dg", "dW_gu", "dW_d"):
        assert np.max(np.abs(fused[k] - plain[k])) <= 1e-11 * np.max(np.abs(plain[k])), k
    np.testing.assert_allclose(fused["e"], fwd["r"][:, None] * plain["dZ"], rtol=1e-13)


# ----------------------------------------------------------------- chains / metric
def test_tiny_chain_matches_block_pieces():
    rng = np.random.default_rng(5)
    X, R = rng.normal(size=(4, 16)), rng.normal(size=(4, 16))
    W1, W2 = rng.normal(size=(16, 16)), rng.normal(size=(16, 8))
    g = 1 + 0.1 * rng.normal(size=16)
    out = O.tiny_chain(X, R, W1, W2, g, 1e-6)["out"]
    # [in, out] weights: the same chain as linear() with the transposes
    h = O.linear(X, W1.T) + R
    ref = O.rms_scale(h, 1e-6)[:, None] * O.linear(h, O.fold_gain(W2.T, g))
    np.testing.assert_allclose(out, ref, rtol=1e-12)


def test_qkv_rope_chain_is_norm_then_gemm_then_rotate():
    rng = np.random.default_rng(6)
    h = rng.normal(size=(8, 16))
    W = rng.normal(size=(48, 16))
    g = 1 + 0.1 * rng.normal(size=16)
    res = O.qkv_rope(h, g, W, 1e-6, seq_len=4, n_rot_cols=32, head_dim=8, base=500000.0)
    # rows 0 and 4 share position 0 -> unrotated
    y = O.rmsnorm(h, g, 1e-6) @ W.T
    np.testing.assert_allclose(res["out"][0], y[0], rtol=1e-13)
    np.testing.assert_allclose(res["out"][4], y[4], rtol=1e-13)
    np.testing.assert_array_equal(res["out"][:, 32:], res["Z"][:, 32:])


def test_mlp_fp8_unit_scales_reduce_to_block_pieces():
    rng = np.random.default_rng(9)
    h = rng.normal(size=(6, 16))
    Xq = O.e4m3_round(h)
    Wq = O.e4m3_round(rng.normal(size=(8, 16)))
    Wdq = O.e4m3_round(rng.normal(size=(16, 4)))
    res = O.mlp_fp8(h, Xq, 1.0, Wq, 1.0, Wdq, 1.0, 1.0, 1e-6, 8)
    r = O.rms_scale(h, 1e-6)
    Z = r[:, None] * (Xq @ Wq.T)
    a = O.swiglu(Z[:, :4], Z[:, 4:])
    np.testing.assert_allclose(res["a"], a, rtol=1e-13)
    np.testing.assert_allclose(res["Y"], O.e4m3_round(a) @ Wdq.T + h, rtol=1e-13)
    assert res["amax"] == np.max(np.abs(a))


def test_mlp_fp8_power_of_two_scales_are_exact():
    # Scaling laws fixed by the arithmetic, exact for powers of two in e4m3's normal range:
    # s_x and s_w enter only as their product; doubling s_wd doubles Y - h; doubling s_a leaves
    # Y unchanged (e4m3(a / 2 s_a) 2 s_a = e4m3(a / s_a) s_a while a / s_a stays normal).
    # Data built to stay there: |h| = 1 (r = 1 / sqrt(1 + eps)), X's codes all 1 and W's codes in
    # [1, 4] with 32 per row, so G and U lie in [1, 4] and a / s_a in [5.8, 126].
    rng = np.random.default_rng(19)
    h = rng.choice([-1.0, 1.0], size=(6, 32))
    Xq = np.ones((6, 32))
    Wq = rng.choice([1.0, 1.5, 2.0, 2.5, 3.0, 3.5, 4.0], size=(16, 32))
    Wdq = O.e4m3_round(rng.normal(size=(32, 8)) * 4)
    run = lambda s_x, s_w, s_wd, s_a: O.mlp_fp8(h, Xq, s_x, Wq, s_w, Wdq, s_wd, s_a, 1e-6, 16)
    base = run(0.25, 0.125, 0.0625, 2.0 ** -3)
    a_over = np.abs(base["a"]) / 2.0 ** -3
    assert np.all((a_over > 2.0 ** -5) & (a_over < 224)), "test data left the normal range"
    np.testing.assert_array_equal(run(0.5, 0.0625, 0.0625, 2.0 ** -3)["Y"], base["Y"])
    np.testing.assert_allclose(run(0.25, 0.125, 0.125, 2.0 ** -3)["Y"] - h, 2 * (base["Y"] - h), rtol=1e-13)
    np.testing.assert_allclose(run(0.25, 0.125, 0.0625, 2.0 ** -2)["Y"], base["Y"], rtol=1e-15)
    assert not np.allclose(run(0.5, 0.125, 0.0625, 2.0 ** -3)["a"], base["a"])   # s_x does act
    assert not np.allclose(run(0.25, 0.125, 0.0625, 0.3)["Y"], base["Y"])        # s_a does act


# ------------------------------------------------------------------ fp8 MLP backward
def _mlp_loss(h, W, W_d, dY, eps):
    """The gain-free MLP forward in exact arithmetic, written out here independently of the
    oracle (x = h, no quantisation), and its loss sum(Y * dY)."""
    r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
    Z = r[:, None] * (h @ W.T)
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    a = G / (1.0 + np.exp(-G)) * U
    return float(np.sum((a @ W_d.T + h) * dY)), Z, a, r


def test_mlp_fp8_backward_identity_quantiser_matches_finite_differences():
    eps = 1e-6
    rng = np.random.default_rng(11)
    h, W, W_d = rng.normal(size=(3, 8)), 0.5 * rng.normal(size=(8, 8)), 0.5 * rng.normal(size=(8, 4))
    dY = rng.normal(size=(3, 8))
    _, Z, a, r = _mlp_loss(h, W, W_d, dY, eps)
    got = O.mlp_fp8_backward(h, h, 1.0, W, 1.0, W_d, 1.0, Z, a, 1.0, r, dY, 1.0, 1.0,
                             quant=lambda v: np.asarray(v, float))
    args = {"h": h, "W": W, "W_d": W_d}
    for name, key in (("h", "dh"), ("W", "dW"), ("W_d", "dW_d")):
        fd = np.zeros_like(args[name])
        for ix in np.ndindex(fd.shape):
            p = {k: v.copy() for k, v in args.items()}
            m = {k: v.copy() for k, v in args.items()}
            p[name][ix] += 1e-6
            m[name][ix] -= 1e-6
            fd[ix] = (_mlp_loss(p["h"], p["W"], p["W_d"], dY, eps)[0] -
                      _mlp_loss(m["h"], m["W"], m["W_d"], dY, eps)[0]) / 2e-6
        err = np.max(np.abs(got[key] - fd)) / np.max(np.abs(fd))
        assert err <= 1e-6, (key, err)


def _fp8_bwd_case(seed=12, M=8, H=16, F=8):
    rng = np.random.default_rng(seed)
    return dict(h=rng.normal(size=(M, H)), Xq_val=O.e4m3_round(rng.normal(size=(M, H)) * 40), s_x=2.0 ** -5,
                Wq_val=O.e4m3_round(rng.normal(size=(2 * F, H)) * 40), s_w=2.0 ** -7,
                Wdq_val=O.e4m3_round(rng.normal(size=(H, F)) * 40), s_wd=2.0 ** -6,
                Z=rng.normal(size=(M, 2 * F)), aq_val=O.e4m3_round(rng.normal(size=(M, F)) * 40), s_a=2.0 ** -4,
                r=0.5 + rng.random(M), dY=rng.normal(size=(M, H)), s_dy=0.011, s_e=0.0023)


def test_mlp_fp8_backward_power_of_two_rescaling_is_exact():
    # doubling dY with s_dy and s_e keeps every e4m3 code and doubles every gradient exactly
    b = _fp8_bwd_case()
    base = O.mlp_fp8_backward(**b)
    d = dict(b, dY=2 * b["dY"], s_dy=2 * b["s_dy"], s_e=2 * b["s_e"])
    dbl = O.mlp_fp8_backward(**d)
    np.testing.assert_array_equal(dbl["dYq_val"], base["dYq_val"])
    np.testing.assert_array_equal(dbl["eq_val"], base["eq_val"])
    for k in ("dA", "e", "c", "t", "dh", "dW_d", "dW"):
        np.testing.assert_array_equal(dbl[k], 2 * base[k], err_msg=k)


def test_mlp_fp8_backward_quantises_like_the_library_cast():
    b = _fp8_bwd_case(seed=13)
    b["s_dy"] = float(np.max(np.abs(b["dY"]))) / 400.0
    e = O.mlp_fp8_backward(**b)["e"]
    b["s_e"] = float(np.max(np.abs(e))) / 400.0
    res = O.mlp_fp8_backward(**b)
    cast = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(res["dYq_val"], cast(b["dY"] / b["s_dy"]))
    np.testing.assert_array_equal(res["eq_val"], cast(res["e"] / b["s_e"]))


def test_mlp_fp8_backward_zero_operands_give_closed_forms():
    b = _fp8_bwd_case(seed=14)
    res = O.mlp_fp8_backward(**dict(b, Xq_val=np.zeros_like(b["Xq_val"])))
    assert np.all(res["dW"] == 0)                       # weight gradient of a zero input
    res = O.mlp_fp8_backward(**dict(b, aq_val=np.zeros_like(b["aq_val"])))
    assert np.all(res["dW_d"] == 0)
    res = O.mlp_fp8_backward(**dict(b, Wdq_val=np.zeros_like(b["Wdq_val"])))
    assert np.all(res["e"] == 0) and np.all(res["dW"] == 0) and np.all(res["c"] == 0)
    np.testing.assert_array_equal(res["dh"], b["dY"])   # only the residual path is left


def test_max_rel_err_floor():
    ref = np.array([0.0, 1.0, -1.0, 1e-9])
    got = ref + np.array([0.01, 0.0, 0.0, 0.01])
    # the floor rms(ref) ~ 0.707 keeps the near-zero entries from dominating
    assert abs(O.max_rel_err(got, ref) - 0.01 / math.sqrt(0.5)) < 1e-9


# ---------------------------------------------------------------------- cross-entropy
def test_logsumexp_matches_scipy_and_closed_forms():
    from scipy.special import logsumexp as lse_lib
    z = RNG.normal(size=(7, 50)) * 10
    np.testing.assert_allclose(O.logsumexp(z), lse_lib(z, axis=1), rtol=1e-14)
    V = 128
    np.testing.assert_allclose(O.logsumexp(np.zeros((2, V))), math.log(V), rtol=1e-15)
    big = np.array([[1000.0, 1000.0]])       # shift makes it finite: 1000 + log 2
    np.testing.assert_allclose(O.logsumexp(big), 1000.0 + math.log(2.0), rtol=1e-15)


def test_cross_entropy_closed_forms():
    V = 64
    ce = O.cross_entropy(np.zeros((3, V)), [0, 5, 63])
    np.testing.assert_allclose(ce["loss"], math.log(V), rtol=1e-15)   # uniform logits
    z = np.full((1, 4), -50.0)
    z[0, 2] = 50.0
    assert O.cross_entropy(z, [2])["loss"][0] < 1e-40                 # confident and right
    np.testing.assert_allclose(O.cross_entropy(z, [0])["loss"][0], 100.0, rtol=1e-12)


def test_xent_partials_combine_to_logsumexp():
    z = RNG.normal(size=(9, 700)) * 5
    for bn in (32, 256, 700, 100):
        m, s = O.xent_partials(z, bn)
        np.testing.assert_allclose(O.xent_combine(m, s), O.logsumexp(z), rtol=1e-13)


def _lm_head_case(M=5, d=8, V=11, seed=4):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(M, d)), 1 + 0.1 * rng.normal(size=d), rng.normal(size=(V, d)) / 2,
            rng.integers(0, V, size=M))


def test_lm_head_xent_backward_matches_finite_differences():
    h, g, W, t = _lm_head_case()
    eps = 1e-6
    f = O.lm_head_xent_forward(h, g, W, t, eps)
    b = O.lm_head_xent_backward(f, h, g, W, t, dloss=1.7)

    def loss(hh, gg, WW):
        return 1.7 * O.lm_head_xent_forward(hh, gg, WW, t, eps)["mean"]

    for name, arr, an in (("h", h, b["dh"]), ("g", g, b["dg"]), ("W", W, b["dW_v"])):
        num = np.zeros_like(arr)
        for ix in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[ix] += 1e-6
            m[ix] -= 1e-6
            args_p = {"h": (p, g, W), "g": (h, p, W), "W": (h, g, p)}[name]
            args_m = {"h": (m, g, W), "g": (h, m, W), "W": (h, g, m)}[name]
            num[ix] = (loss(*args_p) - loss(*args_m)) / 2e-6
        assert np.max(np.abs(num - an)) / np.max(np.abs(num)) <= 1e-6, name


def test_lm_head_fused_backward_equals_chain_rule_and_rows_sum_to_zero():
    h, g, W, t = _lm_head_case(M=12, d=16, V=40, seed=9)
    f = O.lm_head_xent_forward(h, g, W, t, 1e-6)
    plain = O.lm_head_xent_backward(f, h, g, W, t, dloss=0.5)
    fused = O.lm_head_xent_backward_fused(f, h, g, W, t, dloss=0.5)
    for k in ("dh", "dg", "dW_v"):
        assert np.max(np.abs(fused[k] - plain[k])) <= 1e-12 * np.max(np.abs(plain[k])), k
    np.testing.assert_allclose(np.sum(plain["dlogits"], axis=1), 0.0, atol=1e-15)   # softmax - onehot


# ------------------------------------------------------------------- QKV / RoPE backward
def test_rope_inverse_rotation():
    Z, hd, nh = _rope_setup()
    pos = np.arange(Z.shape[0]) * 11 + 2
    back = O.rope_rotate(O.rope_rotate(Z, pos, hd * nh, hd, 500000.0), -pos, hd * nh, hd, 500000.0)
    np.testing.assert_allclose(back, Z, rtol=1e-13, atol=1e-14)


def _qkv_case(M=6, d=8, N=24, seed=12):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(M, d)), 1 + 0.1 * rng.normal(size=d), rng.normal(size=(N, d)) / 2,
            rng.normal(size=(M, N)))


def test_qkv_rope_backward_matches_finite_differences():
    h, g, W, dout = _qkv_case()
    kw = dict(seq_len=4, n_rot_cols=16, head_dim=8, base=10000.0)
    b = O.qkv_rope_backward(h, g, W, dout, 1e-6, **kw)

    def loss(hh, gg, WW):
        return float(np.sum(O.qkv_rope(hh, gg, WW, 1e-6, **kw)["out"] * dout))

    for name, arr, an in (("h", h, b["dh"]), ("g", g, b["dg"]), ("W", W, b["dW"])):
        num = np.zeros_like(arr)
        for ix in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[ix] += 1e-6
            m[ix] -= 1e-6
            ap = {"h": (p, g, W), "g": (h, p, W), "W": (h, g, p)}[name]
            am = {"h": (m, g, W), "g": (h, m, W), "W": (h, g, m)}[name]
            num[ix] = (loss(*ap) - loss(*am)) / 2e-6
        assert np.max(np.abs(num - an)) / np.max(np.abs(num)) <= 1e-6, name


def test_qkv_rope_fused_backward_equals_chain_rule():
    h, g, W, dout = _qkv_case(M=10, d=16, N=48, seed=13)
    kw = dict(seq_len=4, n_rot_cols=32, head_dim=16, base=500000.0)
    out = O.qkv_rope(h, g, W, 1e-6, **kw)["out"]
    plain = O.qkv_rope_backward(h, g, W, dout, 1e-6, **kw)
    fused = O.qkv_rope_backward_fused(h, g, W, dout, out, 1e-6, **kw)
    for k, pk in (("dh", "dh"), ("dg", "dg"), ("dW", "dW")):
        assert np.max(np.abs(fused[k] - plain[pk])) <= 1e-11 * np.max(np.abs(plain[pk])), k
