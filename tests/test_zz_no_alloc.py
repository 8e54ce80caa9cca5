"""coda_block_forward_noalloc: the block forward chain for callers that cannot allocate
device memory (an operator inside a runtime that owns the whole device memory pool, or a
deployment that forbids allocation after start-up).  It takes no workspace; the chain's
partial sums live in the library's static device array.

Checked here, through the C ABI: two calls in a row (different sizes, so the second call
reuses the array the first one left behind) give exactly the results of coda_block_forward
with a caller-allocated workspace (the same kernels in the same order, so bit for bit; a
stale or missing partial would change r and everything after it), and they also meet the
parity tolerance of the other tests; problems beyond the array's size are refused before
anything is launched.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

import coda_synth as S
from tests.gpu_helpers import TOL_BF16, assert_close, f64, fresh_status

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    return coda


def _prepare(C, M, H, F, seed):
    inp = S.block_inputs(M, H, F, seed=seed)
    d = {k: inp[k].to("cuda").contiguous() for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    Wf = torch.empty_like(d["W_gu"])
    C.coda_fold_gain(d["W_gu"], d["g"], Wf)
    d["Wf"] = Wf
    return d, inp["eps"]


def _outs(M, H, F):
    return dict(h=torch.empty((M, H), dtype=BF, device="cuda"), r=torch.empty((M,), device="cuda"),
                a=torch.empty((M, F), dtype=BF, device="cuda"), Y=torch.empty((M, H), dtype=BF, device="cuda"),
                Yp=torch.empty(((H + 255) // 256, M), device="cuda"))


def _with_workspace(C, d, eps, M, H, F):
    o = _outs(M, H, F)
    ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    C.coda_block_forward(d["O"], d["R"], d["W_o"], d["Wf"], d["W_d"], eps, o["h"], o["r"], o["a"], o["Y"], ws,
                         Y_partials=o["Yp"])
    return o


def _no_alloc(C, d, eps, M, H, F):
    o = _outs(M, H, F)
    C.coda_block_forward_noalloc(d["O"], d["R"], d["W_o"], d["Wf"], d["W_d"], eps, o["h"], o["r"], o["a"], o["Y"],
                                 Y_partials=o["Yp"])
    return o


def test_no_alloc_matches_workspace_entry_point_on_two_calls(C):
    shapes = [(640, 512, 1024, 0), (300, 256, 384, 5)]
    prepared = [(_prepare(C, M, H, F, seed), (M, H, F)) for M, H, F, seed in shapes]
    refs = [_with_workspace(C, d, eps, *mhf) for (d, eps), mhf in prepared]
    torch.cuda.synchronize()
    fresh_status()
    gots = [_no_alloc(C, d, eps, *mhf) for (d, eps), mhf in prepared]   # two calls in a row
    torch.cuda.synchronize()
    fresh_status()
    for ref, got, (M, H, F, _) in zip(refs, gots, shapes):
        for k in ("h", "r", "a", "Y", "Yp"):
            assert torch.equal(got[k], ref[k]), f"{k} differs from the workspace call (M={M}, H={H}, F={F})"
            assert_close(f64(got[k]), f64(ref[k]), TOL_BF16, f"{k} (M={M}, H={H}, F={F})")


def test_no_alloc_refuses_oversized_problems(C):
    # never launched: the size checks come first, so these pointers are not dereferenced
    fake = ctypes.c_void_p(0x10000)

    def io(M, H, F, ws=None):
        return C.CodaBlockFwd(M=M, H=H, F=F, eps=1e-6, O=fake, R=fake, W_o=fake, W_gu=fake, W_d=fake, h=fake, r=fake,
                              a=fake, Y=fake, workspace=ws)

    L = C.lib()
    too_many_rows = C.NOALLOC_MAX_PARTIALS // ((2048 + 255) // 256) + 1
    assert L.coda_block_forward_noalloc(ctypes.byref(io(too_many_rows, 2048, 8192)), None) == C.ERR_SHAPE
    assert L.coda_block_forward_noalloc(ctypes.byref(io(256, 2048, 8192, fake)), None) == C.ERR_SHAPE
    assert L.coda_block_forward_noalloc(None, None) == C.ERR_NULL
