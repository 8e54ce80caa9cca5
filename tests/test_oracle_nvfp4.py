"""Pins for the oracle's NVFP4 functions (reading 9: e2m1 codes, e4m3 block scales over 16
K elements, an fp32 tensor scale).  Each pin fixes the answer without the oracle's own
formula: the value table of the 4-bit format, brute-force nearest-value search, data built
to be exactly representable, error bounds of round-to-nearest, power-of-two equivariance,
and per-block brute-force sums for the block-scaled GEMM.

Source: [KuCoin] "CODA: new research optimizes Transformer training with GEMM-epilogue
programming", section "El impuesto a la pereza" (FP8 and FP4 speed up the matmul, so the
traffic around it weighs more)."""
import itertools

import numpy as np

import oracle as O

# the e2m1 magnitudes by code 0..7: sign | exponent (2 bits, bias 1) | mantissa (1 bit)
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _nearest_e2m1(y):
    """Brute force: the table entry nearest to y (ties: the even code), saturating at 6."""
    a = min(abs(y), 6.0)
    d = [abs(a - v) for v in E2M1_TABLE]
    best = min(d)
    cands = [i for i, di in enumerate(d) if di == best]
    code = [i for i in cands if i % 2 == 0][0] if len(cands) > 1 else cands[0]
    return float(np.copysign(E2M1_TABLE[code], y))


# ------------------------------------------------------------------------------ e2m1
def test_e2m1_decode_is_the_format_table():
    vals = O.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(vals[:8], E2M1_TABLE)
    np.testing.assert_array_equal(vals[8:], [-v for v in E2M1_TABLE])
    assert np.signbit(vals[8])                      # code 8 is -0


def test_e2m1_encode_round_trips_every_code():
    codes = np.arange(16)
    np.testing.assert_array_equal(O.e2m1_encode(O.e2m1_decode(codes)), codes)


def test_e2m1_round_is_the_nearest_value_with_ties_to_even():
    grid = np.concatenate([np.arange(-8.0, 8.0, 1 / 64), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 1e9, -1e9]])
    for y in grid:
        assert O.e2m1_round(y) == _nearest_e2m1(y), y
    # the ties themselves, by hand: each goes to the even code
    assert [float(O.e2m1_round(t)) for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 1, 1, 2, 2, 4, 4]


# ------------------------------------------------------------------- quantiser
def test_nvfp4_exactly_representable_blocks_round_trip():
    rng = np.random.default_rng(21)
    R, K = 6, 64
    s = 2.0 ** -7
    sf = 2.0 ** rng.integers(-4, 5, size=(R, K // 16)).astype(float)    # e4m3 powers of two
    q = rng.choice(E2M1_TABLE, size=(R, K)) * rng.choice([-1.0, 1.0], size=(R, K))
    q.reshape(R, K // 16, 16)[:, :, 0] = 6.0                             # every block's amax is 6 sf s
    x = s * np.repeat(sf, 16, axis=1) * q
    q2, sf2 = O.nvfp4_quantize(x, s)
    np.testing.assert_array_equal(sf2, sf)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(O.nvfp4_dequantize(q2, sf2, s), x)


def test_nvfp4_error_is_within_half_a_step():
    rng = np.random.default_rng(22)
    x = (rng.normal(size=(32, 128)) * 3.0).astype(np.float32).astype(float)
    s = float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    q, sf = O.nvfp4_quantize(x, s)
    d = s * np.repeat(sf, 16, axis=1)
    y = x / d
    # spacing of e2m1 at |y|: 0.5 below 2, 1 below 4, 2 above; beyond 6 the error is the overshoot
    step = np.where(np.abs(y) < 2, 0.5, np.where(np.abs(y) < 4, 1.0, 2.0))
    err = np.abs(O.nvfp4_dequantize(q, sf, s) - x) / d
    allowed = np.where(np.abs(y) <= 6, 0.5 * step, np.abs(y) - 6) * (1 + 1e-6) + 1e-6
    assert np.all(err <= allowed)
    # every block scale is amax / 6 to within e4m3's relative half step (1/16)
    amax = np.max(np.abs(x.reshape(32, 8, 16)), axis=2)
    assert np.all(np.abs(sf * 6 * s - amax) <= amax / 16 * (1 + 1e-6))


def test_nvfp4_zero_and_single_value_blocks():
    s = 0.5
    x = np.zeros((2, 32))
    x[1, 20] = -3.0                                  # second row: block 1 holds one value
    q, sf = O.nvfp4_quantize(x, s)
    assert sf[0, 0] == 0 and sf[0, 1] == 0 and sf[1, 0] == 0
    np.testing.assert_array_equal(q[0], 0)
    assert sf[1, 1] == 1.0                          # 3 / (6 * 0.5) = 1 exactly
    assert q[1, 20] == -6.0 and np.count_nonzero(q[1]) == 1


def test_nvfp4_power_of_two_equivariance_and_sign_symmetry():
    rng = np.random.default_rng(23)
    x = rng.normal(size=(8, 64))
    s = 2.0 ** -9
    q, sf = O.nvfp4_quantize(x, s)
    q2, sf2 = O.nvfp4_quantize(x * 8.0, s * 8.0)     # both scaled: the same codes and block scales
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(sf2, sf)
    q3, sf3 = O.nvfp4_quantize(x, s * 4.0)           # only s scaled: block scales shrink 4x
    np.testing.assert_array_equal(q3, q)
    np.testing.assert_array_equal(sf3, sf / 4.0)
    qn, sfn = O.nvfp4_quantize(-x, s)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sfn, sf)


def test_nvfp4_blocks_are_16_consecutive_elements_of_a_row():
    # a large value in one block raises that block's scale only
    x = np.ones((3, 64))
    x[1, 37] = 100.0                                 # row 1, block 2 (elements 32..47)
    q, sf = O.nvfp4_quantize(x, 1.0)
    big = sf[1, 2]
    assert big > 1.0
    others = np.delete(sf.ravel(), 1 * 4 + 2)
    assert np.all(others == others[0]) and others[0] < big


# ------------------------------------------------------------ block-scaled GEMM
def test_block_scaled_gemm_is_the_sum_of_per_block_products():
    rng = np.random.default_rng(24)
    M, N, K = 3, 4, 48
    qa = rng.choice(E2M1_TABLE, size=(M, K)) * rng.choice([-1.0, 1.0], size=(M, K))
    qb = rng.choice(E2M1_TABLE, size=(N, K)) * rng.choice([-1.0, 1.0], size=(N, K))
    sfa = rng.choice([0.25, 0.5, 1.0, 2.0, 3.0], size=(M, K // 16))
    sfb = rng.choice([0.25, 0.5, 1.0, 2.0, 3.0], size=(N, K // 16))
    sa, sb = 0.75, 1.25
    got = O.linear(O.nvfp4_dequantize(qa, sfa, sa), O.nvfp4_dequantize(qb, sfb, sb))
    ref = np.zeros((M, N))
    for m, n, b in itertools.product(range(M), range(N), range(K // 16)):
        ref[m, n] += sa * sb * sfa[m, b] * sfb[n, b] * sum(qa[m, k] * qb[n, k] for k in range(16 * b, 16 * b + 16))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_mlp_nvfp4_unit_scales_reduce_to_block_pieces():
    rng = np.random.default_rng(25)
    M, H, F = 6, 32, 16
    h = rng.normal(size=(M, H))
    one = lambda r, c: np.ones((r, c // 16))
    Xq = O.e2m1_round(h * 2)
    Wq = O.e2m1_round(rng.normal(size=(2 * F, H)) * 2)
    Wdq = O.e2m1_round(rng.normal(size=(H, F)) * 2)
    r = O.rms_scale(h, 1e-6)
    Z = r[:, None] * (Xq @ Wq.T)
    a = O.swiglu(Z[:, :F], Z[:, F:])
    s_a = 2.0 ** np.ceil(np.log2(np.max(np.abs(a)) / (6 * 448)))   # no block scale saturates
    res = O.mlp_nvfp4(h, Xq, one(M, H), 1.0, Wq, one(2 * F, H), 1.0, Wdq, one(H, F), 1.0, s_a, 1e-6, 16)
    np.testing.assert_allclose(res["a"], a, rtol=1e-13)
    assert res["amax"] == np.max(np.abs(a))
    # the SwiGLU output goes through the quantiser before the down GEMM
    aq, asf = O.nvfp4_quantize(a, s_a)
    np.testing.assert_allclose(res["Y"], (s_a * np.repeat(asf, 16, axis=1) * aq) @ Wdq.T + h, rtol=1e-13)
    # 4-bit: each element within a sixth of its block's amax (half the top step 2 of 6),
    # plus the block scale's e4m3 rounding
    err = np.abs(s_a * np.repeat(asf, 16, axis=1) * aq - a)
    bmax = np.repeat(np.max(np.abs(a).reshape(M, F // 16, 16), axis=2), 16, axis=1)
    assert np.all(err <= bmax / 6 * (1 + 1 / 16) + 1e-12)


def test_mlp_nvfp4_power_of_two_scales_are_exact():
    # Scaling laws fixed by the arithmetic, exact for powers of two while block scales stay
    # normal e4m3 numbers: s_x and s_w enter only as their product; doubling s_wd doubles Y - h;
    # doubling s_a halves a's block scales and leaves its codes and Y unchanged.
    rng = np.random.default_rng(26)
    M, H, F = 6, 64, 32
    h = rng.normal(size=(M, H))
    Xq, Xsf = O.nvfp4_quantize(h, 2.0 ** -6)
    Wq, Wsf = O.nvfp4_quantize(rng.normal(size=(2 * F, H)), 2.0 ** -7)
    Wdq, Wdsf = O.nvfp4_quantize(rng.normal(size=(H, F)), 2.0 ** -7)
    run = lambda s_x, s_w, s_wd, s_a: O.mlp_nvfp4(h, Xq, Xsf, s_x, Wq, Wsf, s_w, Wdq, Wdsf, s_wd, s_a, 1e-6, 16)
    a = run(2.0 ** -6, 2.0 ** -7, 2.0 ** -7, 1.0)["a"]
    s_a = 2.0 ** np.round(np.log2(np.max(np.abs(a)) / (6 * 64)))      # block scales near 64 and below
    base = run(2.0 ** -6, 2.0 ** -7, 2.0 ** -7, s_a)
    twice = run(2.0 ** -6, 2.0 ** -7, 2.0 ** -7, 2 * s_a)
    nz = base["asf"] > 0
    assert np.all(base["asf"][nz] >= 2.0 ** -5), "test data left the normal e4m3 range"
    np.testing.assert_array_equal(run(2.0 ** -5, 2.0 ** -8, 2.0 ** -7, s_a)["Y"], base["Y"])
    np.testing.assert_allclose(run(2.0 ** -6, 2.0 ** -7, 2.0 ** -6, s_a)["Y"] - h, 2 * (base["Y"] - h), rtol=1e-13)
    np.testing.assert_array_equal(twice["aq"], base["aq"])
    np.testing.assert_array_equal(twice["asf"], base["asf"] / 2)
    np.testing.assert_array_equal(twice["Y"], base["Y"])
    assert not np.allclose(run(2.0 ** -5, 2.0 ** -7, 2.0 ** -7, s_a)["a"], base["a"])   # s_x does act


def test_nvfp4_quantize_is_the_brute_force_nearest_definition():
    # The plain float64 definition, by brute force over the two value tables: the block scale
    # is the e4m3 value nearest to amax / (6 s) (torch's e4m3 decoding of all 256 bytes; ties to
    # the even code, saturating at 448), and each code is the e2m1 value nearest to x / (sf s).
    import torch
    tab = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()[:127]
    codes = np.arange(127)

    def nearest_e4m3(u):
        d = np.abs(np.minimum(u, 448.0) - tab)
        best = np.flatnonzero(d == d.min())
        return tab[best[0] if len(best) == 1 else [c for c in codes[best] if c % 2 == 0][0]]

    rng = np.random.default_rng(27)
    R, K = 5, 96
    x = rng.normal(size=(R, K)) * np.exp(rng.normal(size=(R, 1)) * 2)
    x[0, :16] = 0.0
    s = float(np.float32(np.max(np.abs(x)) / (6 * 448) * 0.37))     # some blocks saturate at 448
    q, sf = O.nvfp4_quantize(x, s)
    for i in range(R):
        for b in range(K // 16):
            blk = x[i, 16 * b:16 * b + 16]
            want_sf = nearest_e4m3(np.max(np.abs(blk)) / (6.0 * s))
            assert sf[i, b] == want_sf, (i, b)
            for j, v in enumerate(blk):
                want = _nearest_e2m1(v / (want_sf * s)) if want_sf > 0 else 0.0
                assert q[i, 16 * b + j] == want, (i, b, j)
