"""Failure detection on the GPU without a fault: a wait that runs out.

The test hook makes the producer of the next GEMM launch drop one k-block, so the MMA
thread waits for a stage that never fills.  The bounded wait gives up after the watchdog
limit (200 ms here), the kernel leaves through its abort path (drains its copies, frees
TMEM, returns) and the host reads CODA_ERR_DEVICE_TIMEOUT with the site of the wait.
Nothing traps.  The context must still be usable afterwards: the next GEMM is exact."""
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
    assert site in (1, 2, 3, 4, 5), site
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
