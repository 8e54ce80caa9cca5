"""GPU parity of the light row-wise and element-wise entry points, called on their own
through the C ABI: the RMSNorm split r, u = X * g (coda_rms_gain), the RoPE-backward pass
(coda_rope_backward), the gain fold on fp32 weights (coda_fold_gain) and the SM count.

Tolerances come from the arithmetic of each kernel: an fp32 sum of d terms is within
d * 2^-24 of its magnitude sum (Higham's gamma_d), a product rounded once to bf16 (8
significant bits) is within 2^-8 relative, and a product of two fp32 values rounded to fp32
is the oracle's fp64 product rounded to fp32, bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_helpers import TOL_BF16, assert_close, assert_e4m3_codes, f64, fresh_status, seeded

pytestmark = pytest.mark.gpu

BF = torch.bfloat16
U32 = 2.0 ** -24
BASE = 500000.0


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def _padded(M, N, pad, seed, dtype=BF, **kw):
    """A seeded [M, N] view of an [M, N + pad] buffer (row stride above the width)."""
    buf = seeded((M, N + pad), seed, dtype=dtype, **kw).cuda()
    return buf[:, :N]


# ------------------------------------------------------------------------- rms_gain
@pytest.mark.parametrize("M,d,pad", [(1, 8, 0), (300, 520, 0), (77, 4096, 8), (1030, 256, 24)])
def test_rms_gain(C, M, d, pad):
    X = _padded(M, d, pad, 70)
    X[M // 2].zero_()                                  # an all-zero row: r = 1 / sqrt(eps)
    g = seeded((d,), 71, std=0.1, mean=1.0).cuda()
    eps = 1e-5
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    u = torch.empty((M, d), dtype=BF, device="cuda")
    C.coda_rms_gain(X, g, eps, r, u)
    torch.cuda.synchronize()
    fresh_status()
    x = f64(X)
    r_ref = O.rms_scale(x, eps)
    # fp32 sum of d squares, then rsqrt (a few ulp): relative error of r at most half the sum's
    np.testing.assert_allclose(f64(r), r_ref, rtol=d * U32 / 2 + 8 * U32)
    assert f64(r)[M // 2] == pytest.approx(1 / np.sqrt(eps), rel=8 * U32)
    # u = bf16(fp32(x * g)): one bf16 rounding (2^-8) after one fp32 rounding
    u_ref = x * f64(g)[None, :]
    err = np.abs(f64(u) - u_ref)
    assert np.all(err <= np.abs(u_ref) * (2.0 ** -8 + U32) * (1 + 1e-12)), "u = X * g"


def test_rms_gain_matches_the_norm_it_splits(C):
    # r * u is the RMSNorm output y = r h g
    M, d = 257, 1024
    X = seeded((M, d), 72, std=3.0, dtype=BF).cuda()
    g = seeded((d,), 73, std=0.2, mean=1.0).cuda()
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    u = torch.empty((M, d), dtype=BF, device="cuda")
    C.coda_rms_gain(X, g, 1e-6, r, u)
    torch.cuda.synchronize()
    assert_close(f64(r)[:, None] * f64(u), O.rmsnorm(f64(X), f64(g), 1e-6), TOL_BF16, "r u = rmsnorm(X, g)")


# -------------------------------------------------------------------- rope_backward
@pytest.mark.parametrize("M,N,hd,ncols,seq,pad", [
    (300, 768, 64, 640, 100, 0),        # Q and K heads rotated, V copied; ragged rows
    (5, 136, 8, 128, 3, 0),             # the narrowest head, a 17-step row (ragged lane loop)
    (64, 256, 128, 0, 16, 0),           # nothing rotated: e = r dout
    (129, 512, 128, 512, 7, 16),        # everything rotated; padded rows
    (1, 1024, 64, 1024, 1, 0),          # one row at position 0: no rotation at all
])
def test_rope_backward(C, M, N, hd, ncols, seq, pad):
    H = 1024
    dout = _padded(M, N, pad, 74)
    out = _padded(M, N, pad, 75)
    r = seeded((M,), 76, std=0.2, mean=1.0).cuda()
    cos = torch.empty((seq, hd // 2), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, BASE, cos, sin)
    e = torch.empty((M, N), dtype=BF, device="cuda")
    c = torch.empty(M, dtype=torch.float32, device="cuda")
    C.coda_rope_backward(dout, out, r, cos, sin, seq, hd, ncols, H, e, c)
    torch.cuda.synchronize()
    fresh_status()
    d, o, rr = f64(dout), f64(out), f64(r)
    pos = np.arange(M) % seq
    e_ref = rr[:, None] * O.rope_rotate(d, -pos, ncols, hd, BASE)
    assert_close(f64(e), e_ref, TOL_BF16, "e = r R(-phi) dout")
    if ncols == 0 or seq == 1:
        # no rotation: each element is r * dout rounded to fp32, then to bf16
        assert np.all(np.abs(f64(e) - e_ref) <= np.abs(e_ref) * (2.0 ** -8 + U32) * (1 + 1e-12)), "e = r dout"
    p = d * o
    c_ref = rr ** 2 * p.sum(axis=1) / H
    bound = rr ** 2 * np.abs(p).sum(axis=1) / H * (N + 4) * U32
    assert np.all(np.abs(f64(c) - c_ref) <= bound), "c = r^2 sum dout out / H"


def test_rope_backward_inverts_the_forward_rotation(C):
    # R(-phi) R(phi) = I: the backward pass applied to the forward epilogue's rotation of Z
    # gives back r Z (up to the bf16 storage of the rotated tensor)
    M, N, hd, seq = 200, 384, 64, 50
    Z = seeded((M, N), 77, dtype=torch.float64).numpy()
    pos = np.arange(M) % seq
    rotated = torch.from_numpy(O.rope_rotate(Z, pos, N, hd, BASE)).to(BF).cuda()
    r = seeded((M,), 78, std=0.2, mean=1.0).cuda()
    cos = torch.empty((seq, hd // 2), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, BASE, cos, sin)
    e = torch.empty((M, N), dtype=BF, device="cuda")
    c = torch.empty(M, dtype=torch.float32, device="cuda")
    C.coda_rope_backward(rotated, rotated, r, cos, sin, seq, hd, N, 1, e, c)
    torch.cuda.synchronize()
    assert_close(f64(e), f64(r)[:, None] * Z, TOL_BF16, "R(-phi) R(phi) Z")
    # dout = out: c = r^2 |out|^2, every term non-negative
    np.testing.assert_allclose(f64(c), f64(r) ** 2 * np.sum(f64(rotated) ** 2, axis=1), rtol=(N + 4) * U32)


# ------------------------------------------------------------------------ fold_gain
@pytest.mark.parametrize("N,K,pad", [(300, 512, 0), (1, 4, 0), (129, 1000, 12)])
def test_fold_gain_f32_is_the_rounded_exact_product(C, N, K, pad):
    W = _padded(N, K, pad, 79, dtype=torch.float32, std=0.05)
    g = seeded((K,), 80, std=0.1, mean=1.0).cuda()
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    C.coda_fold_gain(W, g, out)
    torch.cuda.synchronize()
    fresh_status()
    # the fp64 product of two fp32 values is exact, so one rounding to fp32 is the answer
    ref = O.fold_gain(f64(W), f64(g)).astype(np.float32)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", [torch.float32, BF])
def test_fold_gain_in_place(C, dtype):
    N, K = 256, 2048
    W = seeded((N, K), 81, std=0.05, dtype=dtype).cuda()
    W0 = f64(W)
    g = seeded((K,), 82, std=0.1, mean=1.0).cuda()
    C.coda_fold_gain(W, g, W)                          # W_out aliases W
    torch.cuda.synchronize()
    ref = O.fold_gain(W0, f64(g))
    if dtype == torch.float32:
        np.testing.assert_array_equal(W.cpu().numpy(), ref.astype(np.float32))
    else:
        assert np.all(np.abs(f64(W) - ref) <= np.abs(ref) * (2.0 ** -8 + U32) * (1 + 1e-12)), "in-place bf16 fold"


@pytest.mark.parametrize("N,K,pad", [(300, 512, 0), (129, 1008, 16)])
def test_fold_gain_e4m3_out_scale(C, N, K, pad):
    """The fold with an FP8 requant: codes of W g / out_scale.  A code is a rounding decision the
    kernel takes in fp32 (W g rounded once, then times the rounded reciprocal: within 3 fp32
    roundings), so each must lie in the e4m3 rounding window of the fp64 value within 1e-6
    relative and almost all must equal its rounding; values beyond 448 saturate."""
    W = _padded(N, K, pad, 83, dtype=BF, std=0.05)
    g = seeded((K,), 84, std=0.1, mean=1.0).cuda()
    ref = O.fold_gain(f64(W), f64(g))
    out_scale = float(np.float32(np.max(np.abs(ref)) / 448.0 * 0.8))   # the largest few saturate
    Q = torch.full((N, K), 0xEE, dtype=torch.uint8, device="cuda")
    C.coda_fold_gain(W, g, Q, out_scale=out_scale)
    torch.cuda.synchronize()
    fresh_status()
    assert_e4m3_codes(Q.cpu().numpy(), ref / out_scale, "W g / out_scale codes", rel=1e-6)
    assert np.any(np.abs(O.e4m3_decode(Q.cpu().numpy())) == 448.0), "no value reached the saturation"


def test_fold_gain_out_scale_divides_bf16_and_fp32(C):
    N, K = 256, 512
    g = seeded((K,), 86, std=0.1, mean=1.0).cuda()
    for dtype in (torch.float32, BF):
        W = seeded((N, K), 85, std=0.05, dtype=dtype).cuda()
        out = torch.empty((N, K), dtype=dtype, device="cuda")
        C.coda_fold_gain(W, g, out, out_scale=0.25)      # a power of two: the reciprocal is exact
        torch.cuda.synchronize()
        ref = O.fold_gain(f64(W), f64(g)) / 0.25
        if dtype == torch.float32:
            np.testing.assert_array_equal(out.cpu().numpy(), ref.astype(np.float32))
        else:
            assert np.all(np.abs(f64(out) - ref) <= np.abs(ref) * (2.0 ** -8 + U32) * (1 + 1e-12))
    fresh_status()


# ------------------------------------------------------------------------- sm count
def test_device_sm_count(C):
    assert C.coda_device_sm_count() == torch.cuda.get_device_properties(0).multi_processor_count
