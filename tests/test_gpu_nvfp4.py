"""GPU parity of the NVFP4 path against the fp64 oracle, through the C ABI (oracle reading 9:
e2m1 codes, e4m3 block scales per 16 K elements, fp32 tensor scales):

* the quantiser: codes and block scales within the rounding window of the oracle's plain
  float64 definition, almost all equal to it;
* the block-scaled GEMM (plain store), on operands the oracle quantised, at ragged sizes;
* the gate/up GEMM with r, SwiGLU and a bf16 or NVFP4 output (codes checked against the
  oracle's rounding window, block scales and amax);
* the down GEMM with the residual and partial sums of squares;
* the whole NVFP4 MLP chain, small and at the LLaMA-3-8B shape on sampled rows.

Source: [KuCoin] "CODA: new research optimizes Transformer training with GEMM-epilogue
programming", section "El impuesto a la pereza" (FP8 and FP4 speed up the matmul)."""
import numpy as np
import pytest
import torch

import oracle as O
from tests import nvfp4_layout as L
from tests.gpu_helpers import TOL_BF16, TOL_FP8, assert_close, dev, f64, fresh_status, nvfp4_window

pytestmark = pytest.mark.gpu
BF = torch.bfloat16
U8 = torch.uint8


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_set_watchdog_ms(2000)
    return coda


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(BF)


def _scale_of(x):
    return float(np.float32(np.max(np.abs(x)) / (6 * 448)))


# ------------------------------------------------------------------------- quantiser
# an fp32 quotient, product and reciprocal each round once (2^-24 relative): 1e-6 covers
# the quantiser's few roundings with room to spare
QUANT_REL = 1e-6


@pytest.mark.parametrize("R,K", [(300, 512), (256, 320), (128, 192)])
def test_quantize_nvfp4_codes_in_rounding_window(C, R, K):
    X = _bf16((R, K), 31 + R)
    X[0, :16] = 0.0                                   # an all-zero block: scale 0, codes 0
    X[1, 5] = 1e4                                     # one large value: its block saturates nothing
    x = f64(X)
    s = _scale_of(x)
    Q = C.Nvfp4.empty(R, K, s)
    Q.scales.fill_(0xEE)                              # padding rows must be overwritten with 0
    amax = torch.zeros((1,), device="cuda")
    C.coda_quantize_nvfp4(dev(X), Q, amax=amax)
    torch.cuda.synchronize()
    fresh_status()
    got_q = O.e2m1_decode(L.unpack_codes(Q.codes.cpu().numpy()))
    buf = Q.scales.cpu().numpy()
    got_sf = O.e4m3_decode(L.from_atoms(buf, R, K))
    same_sf, same_q, ambiguous, _ = nvfp4_window(got_q, got_sf, x, s, QUANT_REL)
    print(f"nvfp4 quantiser {R}x{K}: block scales equal to the oracle's {same_sf:.6f}, codes {same_q:.6f} "
          f"(within fp32 reach of a midpoint: {ambiguous:.6f})")
    # bf16 values over e4m3 block scales often land on an e2m1 midpoint up to the rounding of
    # the fp32 tensor scale: those few ties may round either way (about 0.1% of the codes)
    assert same_sf >= 0.999 and same_q >= 0.995 and ambiguous <= 0.01
    assert np.all(got_sf[0, :1] == 0) and np.all(got_q[0, :16] == 0)
    used = np.zeros(buf.size, dtype=bool)
    used[L.atom_offsets(R, K)] = True
    assert not buf[~used].any(), "scales of padding rows are not zero"
    assert float(amax.item()) == float(np.max(np.abs(x)))


# ------------------------------------------------------------- block-scaled GEMM
@pytest.mark.parametrize("M,N,K", [(300, 384, 512), (1024, 1024, 2048), (128, 128, 256), (1, 128, 256)])
def test_nvfp4_gemm_store(C, M, N, K):
    xa = f64(_bf16((M, K), 41, 2.0))
    xb = f64(_bf16((N, K), 42, 0.05))
    A, qa, sfa = L.oracle_nvfp4(xa, _scale_of(xa))
    B, qb, sfb = L.oracle_nvfp4(xb, _scale_of(xb))
    out = torch.empty((M, N), device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out, tensor_scale=A.s * B.s)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s))
    got = f64(out)
    err = O.max_rel_err(got, ref)
    if err > 1e-3:   # name the rows / columns that disagree, to tell a layout mistake at a glance
        bad = np.abs(got - ref) > 1e-3 * np.sqrt(np.mean(ref ** 2))
        rows, cols = np.nonzero(bad.any(axis=1))[0], np.nonzero(bad.any(axis=0))[0]
        pytest.fail(f"max rel err {err:.3e}; {len(rows)} rows (first {rows[:8]}), {len(cols)} cols (first {cols[:8]})")


def test_nvfp4_gemm_split_k(C):
    """Few tiles and a long K: the fp32 GEMM splits K across CTA pairs and reduce-adds the
    slices into the zeroed output (each slice's MMAs and scale stores start mid-K)."""
    M, N, K = 256, 256, 16384
    xa, xb = f64(_bf16((M, K), 45)), f64(_bf16((N, K), 46, 0.02))
    A, qa, sfa = L.oracle_nvfp4(xa, _scale_of(xa))
    B, qb, sfb = L.oracle_nvfp4(xb, _scale_of(xb))
    out = torch.full((M, N), float("nan"), device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out, tensor_scale=A.s * B.s)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s))
    assert_close(f64(out), ref, 1e-3, "split-K fp32 out")


def test_nvfp4_gemm_bf16_out_and_k_equal_one_stage(C):
    M, N, K = 256, 256, 256
    xa, xb = f64(_bf16((M, K), 43)), f64(_bf16((N, K), 44, 0.02))
    A, qa, sfa = L.oracle_nvfp4(xa, _scale_of(xa))
    B, qb, sfb = L.oracle_nvfp4(xb, _scale_of(xb))
    out = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out, tensor_scale=A.s * B.s)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s))
    assert_close(f64(out), ref, TOL_BF16, "bf16 out")


# --------------------------------------------------------- gate/up + SwiGLU, down
def _swiglu_case(M, H, F, seed):
    h = f64(_bf16((M, H), seed))
    W = f64(_bf16((2 * F, H), seed + 1, 0.015))
    X, qx, sfx = L.oracle_nvfp4(h, _scale_of(h))
    Wq, qw, sfw = L.oracle_nvfp4(W, _scale_of(W))
    r = O.rms_scale(h, 1e-6).astype(np.float32)
    Z = r.astype(np.float64)[:, None] * O.linear(O.nvfp4_dequantize(qx, sfx, X.s), O.nvfp4_dequantize(qw, sfw, Wq.s))
    a = O.swiglu(Z[:, :F], Z[:, F:])
    return h, X, Wq, r, a


def test_nvfp4_swiglu_bf16_out(C):
    M, H, F = 300, 512, 384
    h, X, Wq, r, a = _swiglu_case(M, H, F, 51)
    out = torch.empty((M, F), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(X, Wq, [C.OP_TENSOR_SCALE, C.OP_ROW_SCALE, C.OP_SWIGLU], out,
                         row_scale=torch.from_numpy(r).cuda(), tensor_scale=X.s * Wq.s)
    torch.cuda.synchronize()
    fresh_status()
    assert_close(f64(out), a, TOL_BF16, "a")


def _check_nvfp4_output(out, a, s_a, M, F, rel=1e-4):
    """An NVFP4 output is a set of rounding decisions taken in fp32 on a value that carries the
    GEMM's accumulation error: each block scale and each code must be a rounding neighbour of
    the oracle's value within a relative distance `rel`, almost all must equal the oracle's own
    rounding, and the dequantised tensor must be within half an e2m1 step of a."""
    got_q = O.e2m1_decode(L.unpack_codes(out.codes.cpu().numpy()))
    got_sf = O.e4m3_decode(L.from_atoms(out.scales.cpu().numpy(), M, F))
    same_sf, same_q, ambiguous, _ = nvfp4_window(got_q, got_sf, a, s_a, rel)
    print(f"nvfp4 output {M}x{F}: block scales equal to the oracle's {same_sf:.6f}, codes {same_q:.6f} "
          f"(within {rel:g} of a midpoint: {ambiguous:.6f})")
    assert same_sf >= 0.999 and same_q >= 0.999 and ambiguous <= 0.01
    amax_b = np.max(np.abs(a).reshape(M, F // 16, 16), axis=2)
    deq = L.nvfp4_values(out, M, F)
    bmax = np.repeat(amax_b, 16, axis=1)
    assert np.all(np.abs(deq - a) <= bmax / 6 * (1 + 1 / 16) + rel * bmax + 1e-30)


def test_nvfp4_swiglu_nvfp4_out_codes_scales_amax(C):
    M, H, F = 300, 512, 384
    h, X, Wq, r, a = _swiglu_case(M, H, F, 52)
    s_a = _scale_of(a)
    out = C.Nvfp4.empty(M, F, s_a)
    amax = torch.zeros((1,), device="cuda")
    C.coda_gemm_epilogue(X, Wq, [C.OP_TENSOR_SCALE, C.OP_ROW_SCALE, C.OP_SWIGLU, C.OP_AMAX], out,
                         row_scale=torch.from_numpy(r).cuda(), tensor_scale=X.s * Wq.s, amax=amax)
    torch.cuda.synchronize()
    fresh_status()
    assert abs(float(amax.item()) - np.max(np.abs(a))) <= 1e-3 * np.max(np.abs(a))
    _check_nvfp4_output(out, a, s_a, M, F)


def test_nvfp4_down_gemm_residual_partials(C):
    M, H, F = 300, 512, 768
    a = f64(_bf16((M, F), 61, 0.5))
    Wd = f64(_bf16((H, F), 62, 0.015))
    Hres = _bf16((M, H), 63)
    A, qa, sfa = L.oracle_nvfp4(a, _scale_of(a))
    B, qb, sfb = L.oracle_nvfp4(Wd, _scale_of(Wd))
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE, C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL], Y,
                         residual=dev(Hres), tensor_scale=A.s * B.s, row_partials=P)
    torch.cuda.synchronize()
    fresh_status()
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s)) + f64(Hres)
    assert_close(f64(Y), ref, TOL_BF16, "Y")
    assert_close(f64(P), O.partial_sumsq(f64(Y), 256), 1e-4, "partials of the stored Y")


# ------------------------------------------------------------------------ the chain
def _chain(C, M, H, F, seed):
    h = _bf16((M, H), seed)
    hx = f64(h)
    Wgu = f64(_bf16((2 * F, H), seed + 1, 0.015))
    Wd = f64(_bf16((H, F), seed + 2, 0.015))
    X, qx, sfx = L.oracle_nvfp4(hx, _scale_of(hx))
    Wq, qw, sfw = L.oracle_nvfp4(Wgu, _scale_of(Wgu))
    Wdq, qd, sfd = L.oracle_nvfp4(Wd, _scale_of(Wd))
    return h, hx, (X, qx, sfx), (Wq, qw, sfw), (Wdq, qd, sfd)


def _run_chain(C, h, X, Wq, Wdq, s_a, M, H, F):
    r = torch.empty((M,), device="cuda")
    a = C.Nvfp4.empty(M, F, s_a)
    amax = torch.empty((1,), device="cuda")
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    C.coda_mlp_nvfp4(dev(h), X, Wq, Wdq, 1e-6, r, a, amax, Y, P)
    torch.cuda.synchronize()
    fresh_status()
    return r, a, amax, Y, P


def test_mlp_nvfp4_chain_small(C):
    M, H, F = 300, 512, 768
    h, hx, (X, qx, sfx), (Wq, qw, sfw), (Wdq, qd, sfd) = _chain(C, M, H, F, 71)
    pre = O.mlp_nvfp4(hx, qx, sfx, X.s, qw, sfw, Wq.s, qd, sfd, Wdq.s, 1.0, 1e-6, 256)   # amax of a
    s_a = _scale_of(pre["a"])
    ref = O.mlp_nvfp4(hx, qx, sfx, X.s, qw, sfw, Wq.s, qd, sfd, Wdq.s, s_a, 1e-6, 256)
    r, a, amax, Y, P = _run_chain(C, h, X, Wq, Wdq, s_a, M, H, F)
    assert_close(f64(r), ref["r"], 1e-5, "r")
    assert abs(float(amax.item()) - ref["amax"]) <= 1e-3 * ref["amax"]
    _check_nvfp4_output(a, ref["a"], s_a, M, F)
    assert_close(f64(Y), ref["Y"], TOL_FP8, "Y")
    assert_close(f64(P), O.partial_sumsq(f64(Y), 256), 1e-4, "partials of the stored Y")


def test_mlp_nvfp4_chain_llama8b_shape_sampled_rows(C):
    """M = 16384 tokens, H = 4096, F = 14336: the whole chain on the GPU, the oracle on 96
    sampled rows (rows are independent in the forward)."""
    M, H, F = 16384, 4096, 14336
    h, hx, (X, qx, sfx), (Wq, qw, sfw), (Wdq, qd, sfd) = _chain(C, M, H, F, 81)
    rows = np.concatenate([np.arange(32), np.random.default_rng(5).choice(np.arange(32, M), 64, replace=False)])
    pre = O.mlp_nvfp4(hx[rows], qx[rows], sfx[rows], X.s, qw, sfw, Wq.s, qd, sfd, Wdq.s, 1.0, 1e-6, 256)
    s_a = _scale_of(pre["a"]) * 2.0    # headroom for rows outside the sample
    ref = O.mlp_nvfp4(hx[rows], qx[rows], sfx[rows], X.s, qw, sfw, Wq.s, qd, sfd, Wdq.s, s_a, 1e-6, 256)
    r, a, amax, Y, P = _run_chain(C, h, X, Wq, Wdq, s_a, M, H, F)
    assert_close(f64(r)[rows], ref["r"], 1e-5, "r")
    assert float(amax.item()) >= ref["amax"] * (1 - 1e-3)
    assert_close(f64(Y)[rows], ref["Y"], TOL_FP8, "Y (sampled rows)")
    assert_close(f64(P)[:, rows], O.partial_sumsq(f64(Y)[rows], 256), 1e-4, "partials (sampled rows)")
