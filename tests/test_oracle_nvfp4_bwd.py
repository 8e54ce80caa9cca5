"""Pins for the oracle's NVFP4 MLP backward (reading 10: each backward GEMM quantises its two
operands along its own K).  Nothing here reuses the oracle's formulas:

* without quantisation the gradients are those of the MLP forward by central finite
  differences in fp64;
* with quantisation, every output equals a brute-force evaluation on tiny shapes: block scales
  and codes found by nearest-value search over the e4m3 and e2m1 value tables, blocks of 16
  taken along the axis each GEMM contracts, and the GEMMs as explicit sums;
* planted mistakes (a quantisation along the wrong axis, a dropped term) fail those pins.

Source: [KuCoin] "CODA: new research optimizes Transformer training with GEMM-epilogue
programming", sections "El epílogo esconde un tesoro" (the backward inherits the structure)
and "El impuesto a la pereza" (FP4 operands for the matmul)."""
import itertools

import numpy as np
import pytest
import torch

import oracle as O

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()[:127]


def _nearest(table, y, sat):
    """Nearest entry of a non-negative value table (ties: the entry of even index), with sign."""
    a = min(abs(y), sat)
    d = [abs(a - v) for v in table]
    best = min(d)
    idx = [i for i, di in enumerate(d) if di == best]
    i = idx[0] if len(idx) == 1 else [j for j in idx if j % 2 == 0][0]
    return float(np.copysign(table[i], y))


def _bf_block(vals, s):
    """Brute-force NVFP4 of one block of 16 values: dequantised values."""
    sf = _nearest(list(E4M3), max(abs(v) for v in vals) / (6.0 * s), 448.0)
    if sf == 0:
        return [0.0] * len(vals)
    return [s * sf * _nearest(E2M1, v / (sf * s), 6.0) for v in vals]


def _bf_quant(x, s, axis):
    """x quantised in blocks of 16 along `axis` (1: along a row, 0: along a column)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    R, C = x.shape
    if axis == 1:
        for i, b in itertools.product(range(R), range(C // 16)):
            out[i, 16 * b:16 * b + 16] = _bf_block(list(x[i, 16 * b:16 * b + 16]), s)
    else:
        for j, b in itertools.product(range(C), range(R // 16)):
            out[16 * b:16 * b + 16, j] = _bf_block(list(x[16 * b:16 * b + 16, j]), s)
    return out


def _gemm(A, B):
    """C = A B as explicit sums."""
    A, B = np.asarray(A), np.asarray(B)
    C = np.zeros((A.shape[0], B.shape[1]))
    for i, j in itertools.product(range(A.shape[0]), range(B.shape[1])):
        C[i, j] = sum(A[i, k] * B[k, j] for k in range(A.shape[1]))
    return C


def _tiny(M, H, F, seed):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(M, H))
    W_gu = rng.normal(size=(2 * F, H)) * 0.3
    W_d = rng.normal(size=(H, F)) * 0.3
    dY = rng.normal(size=(M, H))
    return h, W_gu, W_d, dY


def _forward(h, W_gu, W_d, eps):
    r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
    Z = r[:, None] * (h @ W_gu.T)
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    a = G / (1.0 + np.exp(-G)) * U
    return r, Z, a @ W_d.T + h


def test_unquantised_gradients_are_the_finite_differences():
    M, H, F, eps = 5, 8, 4, 1e-6
    h, W_gu, W_d, dY = _tiny(M, H, F, 31)
    r, Z, _ = _forward(h, W_gu, W_d, eps)
    got = O.mlp_nvfp4_backward(h, W_gu, W_d, Z, r, dY, 1, 1, 1, 1, 1, 1, quant=False)
    loss = lambda h_, Wg, Wd: float(np.sum(dY * _forward(h_, Wg, Wd, eps)[2]))
    step = 1e-6
    for name, arr, idx in (("dh", h, 0), ("dW", W_gu, 1), ("dW_d", W_d, 2)):
        fd = np.zeros_like(arr)
        for pos in itertools.product(*map(range, arr.shape)):
            args = [h.copy(), W_gu.copy(), W_d.copy()]
            args[idx][pos] += step
            up = loss(*args)
            args[idx][pos] -= 2 * step
            fd[pos] = (up - loss(*args)) / (2 * step)
        np.testing.assert_allclose(got[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_quantised_gradients_match_brute_force_blocks_along_each_contraction():
    M, H, F, eps = 32, 32, 16, 1e-6
    h, W_gu, W_d, dY = _tiny(M, H, F, 32)
    r, Z, _ = _forward(h, W_gu, W_d, eps)
    sc = lambda x: float(np.max(np.abs(x)) / (6 * 448))
    G, U = Z[:, :F], Z[:, F:]
    a = G / (1.0 + np.exp(-G)) * U
    s_dy, s_a, s_x, s_wt, s_wdt = sc(dY) * 1.5, sc(a), sc(h), sc(W_gu), sc(W_d)
    # e for its delayed scale, by the same formulas without quantisation of e
    dA0 = _gemm(_bf_quant(dY, s_dy, 1), _bf_quant(W_d.T, s_wdt, 1).T)
    sg = 1.0 / (1.0 + np.exp(-G))
    e = r[:, None] * np.hstack([dA0 * U * sg * (1 + G * (1 - sg)), dA0 * G * sg])
    s_e = sc(e) * 1.25
    got = O.mlp_nvfp4_backward(h, W_gu, W_d, Z, r, dY, s_dy, s_e, s_a, s_x, s_wt, s_wdt)
    np.testing.assert_allclose(got["dA"], dA0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["e"], e, rtol=1e-12, atol=1e-12)
    c = r * np.sum(e * Z, axis=1) / H
    np.testing.assert_allclose(got["c"], c, rtol=1e-12)
    t = _gemm(_bf_quant(e, s_e, 1), _bf_quant(W_gu.T, s_wt, 1).T)
    np.testing.assert_allclose(got["dh"], t - c[:, None] * h + dY, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["dW_d"], _gemm(_bf_quant(dY, s_dy, 0).T, _bf_quant(a, s_a, 0)), rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(got["dW"], _gemm(_bf_quant(e, s_e, 0).T, _bf_quant(h, s_x, 0)), rtol=1e-12,
                               atol=1e-12)


def test_round_cols_is_exact_on_column_blocks_and_round_rows_on_row_blocks():
    # values exactly representable with one block scale per 16 rows of a column are kept by
    # the column quantiser, and lose precision in the row quantiser (and the other way round)
    rng = np.random.default_rng(33)
    R, C, s = 32, 32, 2.0 ** -6
    q = rng.choice(E2M1, size=(R, C)) * rng.choice([-1.0, 1.0], size=(R, C))
    q[::16, :] = 6.0                                              # each column block's amax is 6 sf s
    sf = 2.0 ** rng.integers(-3, 4, size=(R // 16, C))
    x = s * np.repeat(sf, 16, axis=0) * q
    np.testing.assert_array_equal(O.nvfp4_round_cols(x, s), x)
    assert not np.array_equal(O.nvfp4_round_rows(x, s), x)
    np.testing.assert_array_equal(O.nvfp4_round_rows(x.T, s), x.T)
