"""Failure detection on the GPU without a fault: a wait that runs out.

The test hook makes the producer of the next GEMM launch drop one k-block (in both CTAs of
a pair, or in one of them only), so the MMA thread waits for a stage that never fills.  The
bounded wait gives up after the watchdog limit (200 ms here), the kernel leaves through its
abort path (drains its copies, frees TMEM, returns) and the host reads
CODA_ERR_DEVICE_TIMEOUT with the site of the wait.  Nothing traps.  The context must still
be usable afterwards: the next GEMM is exact."""
import pytest
import torch

import oracle as O
from tests.gpu_helpers import TOL_BF16, assert_close, dev, f64, seeded

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture()
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    coda.coda_get_device_status()          # start from a clean status word
    yield coda
    coda.coda_inject_dropped_stage(False)
    coda.coda_set_watchdog_ms(2000)


def test_dropped_stage_times_out_and_context_survives(C):
    M, N, K = 256, 512, 512
    A = dev(seeded((M, K), 60, dtype=BF))
    W = dev(seeded((N, K), 61, std=0.05, dtype=BF))
    out = torch.zeros((M, N), dtype=BF, device="cuda")
    C.coda_set_watchdog_ms(200)
    C.coda_inject_dropped_stage(True)
    C.coda_gemm_epilogue(A, W, [], out)
    st, site = C.coda_get_device_status()
    assert st == C.ERR_DEVICE_TIMEOUT, st
    assert site in (1, 2, 3, 4, 5, 6, 7), site
    # the status word is cleared by the read
    st2, site2 = C.coda_get_device_status()
    assert (st2, site2) == (C.OK, 0)
    # the hook fires once; the next call runs normally and is exact
    C.coda_set_watchdog_ms(2000)
    out2 = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(A, W, [], out2)
    st3, _ = C.coda_get_device_status()
    assert st3 == C.OK
    assert_close(f64(out2), O.linear(f64(A), f64(W)), TOL_BF16, "GEMM after a timed-out launch")


@pytest.mark.parametrize("mode,what", [(2, "second CTA only"), (3, "leader only")])
def test_one_side_of_a_pair_drops_a_stage(C, mode, what):
    """A CTA pair whose two producers disagree: with mode 2 the leader arms the k-block's phase
    for both CTAs' bytes and the second CTA never sends its own; with mode 3 the second CTA's
    bytes land on a phase the leader never armed.  Either way the MMA wait runs out, and at
    exit the leader completes that phase for the missing side and waits for every copy to land
    before the pair leaves.  The next launch is exact; so is one with several waves of tiles."""
    M, N, K = 512, 1024, 1024
    A = dev(seeded((M, K), 68, dtype=BF))
    W = dev(seeded((N, K), 69, std=0.05, dtype=BF))
    out = torch.zeros((M, N), dtype=BF, device="cuda")
    C.coda_set_watchdog_ms(200)
    C.coda_inject_dropped_stage(mode)
    C.coda_gemm_epilogue(A, W, [], out)
    st, site = C.coda_get_device_status()
    assert st == C.ERR_DEVICE_TIMEOUT, (what, st)
    assert site in (1, 2, 3, 4, 5, 6, 7), site
    C.coda_set_watchdog_ms(2000)
    out2 = torch.empty((M, N), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(A, W, [], out2)
    assert C.coda_get_device_status()[0] == C.OK
    assert_close(f64(out2), O.linear(f64(A), f64(W)), TOL_BF16, f"GEMM after a timed-out launch ({what})")
    M2, N2 = 4096, 4096                                  # 256 tiles over the resident pairs
    A2 = dev(seeded((M2, K), 70, dtype=BF))
    W2 = dev(seeded((N2, K), 71, std=0.05, dtype=BF))
    out3 = torch.empty((M2, N2), dtype=BF, device="cuda")
    C.coda_gemm_epilogue(A2, W2, [], out3)
    assert C.coda_get_device_status()[0] == C.OK
    assert_close(f64(out3), O.linear(f64(A2), f64(W2)), TOL_BF16, "a multi-wave GEMM afterwards")


def test_inject_mode_out_of_range_is_refused(C):
    with pytest.raises(C.CodaError):
        C.coda_inject_dropped_stage(4)


@pytest.mark.parametrize("program", ["residual", "swiglu_backward"])
def test_dropped_stage_with_side_inputs_in_flight(C, program):
    """The same with epilogue programs whose side inputs (the residual; the saved Z) are
    already being loaded when the wait runs out: the epilogue lets those copies land before
    the CTA exits, and the next launch of the same program is exact."""
    M, N, K = 1024, 1024, 256
    A = dev(seeded((M, K), 62, dtype=BF))
    W = dev(seeded((N, K), 63, std=0.05, dtype=BF))
    if program == "residual":
        R = dev(seeded((M, N), 64, dtype=BF))
        out = torch.zeros((M, N), dtype=BF, device="cuda")
        run = lambda o: C.coda_gemm_epilogue(A, W, [C.OP_ADD_SIDE], o, residual=R)
        ref = lambda: O.linear(f64(A), f64(W)) + f64(R)
    else:
        W = dev(seeded((K, N), 63, std=0.05, dtype=BF)).t()   # read MN-major, as the backward reads W_d
        Z = dev(seeded((M, 2 * N), 65, dtype=BF))
        r = dev(seeded((M,), 66, std=0.1, mean=1.0))
        S_ = torch.empty(((N + 255) // 256, M), device="cuda")
        out = torch.zeros((M, 2 * N), dtype=BF, device="cuda")
        run = lambda o: C.coda_gemm_epilogue(A, W, [C.OP_SWIGLU_BWD, C.OP_ROW_SCALE, C.OP_ROW_DOT_PARTIAL], o,
                                             aux_in=Z, row_scale=r, row_partials=S_)

        def ref():
            dA, z, rr = O.linear(f64(A), f64(W)), f64(Z), f64(r)[:, None]
            G, U = z[:, :N], z[:, N:]
            return rr * __import__("numpy").hstack([dA * U * O.silu_grad(G), dA * O.silu(G)])
    C.coda_set_watchdog_ms(200)
    C.coda_inject_dropped_stage(True)
    run(out)
    st, site = C.coda_get_device_status()
    assert st == C.ERR_DEVICE_TIMEOUT, st
    assert site in (1, 2, 3, 4, 5, 6, 7), site
    C.coda_set_watchdog_ms(2000)
    out2 = torch.empty_like(out)
    run(out2)
    st3, _ = C.coda_get_device_status()
    assert st3 == C.OK
    assert_close(f64(out2), ref(), TOL_BF16, f"{program} after a timed-out launch")


def test_dropped_stage_in_a_block_scaled_nvfp4_gemm(C):
    """The NVFP4 GEMM, whose MMA thread also copies each stage's block scales into TMEM: a
    stage that never fills ends the launch through the abort path, and the next launch is
    exact."""
    import numpy as np
    from tests import nvfp4_layout as L
    M, N, K = 512, 512, 1024
    g = torch.Generator().manual_seed(67)
    xa = f64((torch.randn((M, K), generator=g)).to(BF))
    xb = f64((torch.randn((N, K), generator=g) * 0.05).to(BF))
    sc = lambda x: float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    A, qa, sfa = L.oracle_nvfp4(xa, sc(xa))
    B, qb, sfb = L.oracle_nvfp4(xb, sc(xb))
    out = torch.zeros((M, N), device="cuda")
    C.coda_set_watchdog_ms(200)
    C.coda_inject_dropped_stage(True)
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out, tensor_scale=A.s * B.s)
    st, site = C.coda_get_device_status()
    assert st == C.ERR_DEVICE_TIMEOUT, st
    assert site in (1, 2, 3, 4, 5, 6, 7), site
    C.coda_set_watchdog_ms(2000)
    out2 = torch.empty((M, N), device="cuda")
    C.coda_gemm_epilogue(A, B, [C.OP_TENSOR_SCALE], out2, tensor_scale=A.s * B.s)
    st2, _ = C.coda_get_device_status()
    assert st2 == C.OK
    ref = O.linear(O.nvfp4_dequantize(qa, sfa, A.s), O.nvfp4_dequantize(qb, sfb, B.s))
    assert_close(f64(out2), ref, 1e-3, "NVFP4 GEMM after a timed-out launch")


def test_dropped_stage_in_the_nvfp4_swiglu_output_gemm(C):
    """The NVFP4 SwiGLU with NVFP4 output, whose scale warps also form half of every tile and
    stage the next tile's block scales between their output chunks: a dropped stage (operands
    and scales) ends the launch through the abort path, and the next launch's codes, block
    scales and amax are bit-identical to a launch made before the fault."""
    import numpy as np
    from tests import nvfp4_layout as L
    M, H, F = 4096, 1024, 1024                            # 128 tiles: more than the CTA pairs
    g = torch.Generator().manual_seed(72)
    xh = f64((torch.randn((M, H), generator=g)).to(BF))
    xw = f64((torch.randn((2 * F, H), generator=g) * 0.03).to(BF))
    sc = lambda x: float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    X, _, _ = L.oracle_nvfp4(xh, sc(xh))
    W, _, _ = L.oracle_nvfp4(xw, sc(xw))
    r = dev(seeded((M,), 73, std=0.1, mean=1.0))

    def run():
        out = C.Nvfp4.empty(M, F, 0.01)
        amax = torch.zeros((1,), device="cuda")
        C.coda_gemm_epilogue(X, W, [C.OP_TENSOR_SCALE, C.OP_ROW_SCALE, C.OP_SWIGLU, C.OP_AMAX], out,
                             row_scale=r, tensor_scale=X.s * W.s, amax=amax)
        return out, amax

    ref, ref_amax = run()
    assert C.coda_get_device_status()[0] == C.OK
    C.coda_set_watchdog_ms(200)
    C.coda_inject_dropped_stage(True)
    run()
    st, site = C.coda_get_device_status()
    assert st == C.ERR_DEVICE_TIMEOUT, st
    assert site in (1, 2, 3, 4, 5, 6, 7), site
    C.coda_set_watchdog_ms(2000)
    got, got_amax = run()
    assert C.coda_get_device_status()[0] == C.OK
    assert torch.equal(got.codes, ref.codes) and torch.equal(got.scales, ref.scales)
    assert torch.equal(got_amax, ref_amax)
