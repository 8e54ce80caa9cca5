"""Launch overlap keeps stream order: the chains give the same results with the overlap on
(each kernel launched with a programmatic dependency on the previous one; GEMMs whose operands
the previous kernel does not write stream them before it ends) and off (plain serialisation),
also when a chain is issued many times back to back, where every kernel's outputs are read or
overwritten by its neighbours.  Kernels without split-K are deterministic, so their outputs
must match bit for bit; fp32 weight gradients that a split-K GEMM reduce-adds in any order are
compared to 1e-5."""
import pytest
import torch

import coda_synth as S
from tests.gpu_helpers import dev, fresh_status

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture()
def C():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda
    coda.lib()
    yield coda
    coda.coda_set_launch_overlap(True)


def _block_fwd_bwd(C, d, inp, M, H, F):
    o = {k: torch.empty(s, dtype=BF, device="cuda") for k, s in
         (("h", (M, H)), ("u", (M, H)), ("a", (M, F)), ("Y", (M, H)), ("Z", (M, 2 * F)), ("e", (M, 2 * F)),
          ("dh", (M, H)), ("dO", (M, H)))}
    o.update(r=torch.empty((M,), device="cuda"), c=torch.empty((M,), device="cuda"),
             dW_o=torch.empty((H, H), device="cuda"), dW_gu=torch.empty((2 * F, H), device="cuda"),
             dW_d=torch.empty((H, F), device="cuda"), dg=torch.empty((H,), device="cuda"))
    wsf = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    wsb = torch.empty((C.coda_workspace_size(C.WS_BLOCK_BWD, M, H, F) // 4,), device="cuda")

    def run():
        C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], inp["eps"], o["h"], o["r"], o["a"],
                             o["Y"], wsf, Z=o["Z"], g=d["g"], u=o["u"])
        C.coda_block_backward(d["O"], d["W_o"], d["W_gu"], d["W_d"], d["g"], o["h"], o["r"], o["Z"], o["a"], d["dY"],
                              o["e"], o["dh"], o["dO"], o["dW_o"], o["dW_gu"], o["dW_d"], o["dg"], o["c"], wsb)
    return o, run


def _compare(ref, got):
    for k in ref:
        if k in ("dW_o", "dW_gu", "dW_d", "dg"):
            torch.testing.assert_close(got[k], ref[k], rtol=1e-5, atol=1e-6, msg=k)
        else:
            assert torch.equal(got[k], ref[k]), k


def test_block_chains_same_with_and_without_overlap_and_back_to_back(C):
    M, H, F = 640, 512, 1024
    inp = S.block_inputs(M, H, F, seed=4, with_grad=True)
    d = {k: dev(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    C.coda_set_launch_overlap(False)
    o, run = _block_fwd_bwd(C, d, inp, M, H, F)
    run()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in o.items()}
    C.coda_set_launch_overlap(True)
    for v in o.values():
        v.zero_()
    for _ in range(20):                # 20 x 12 launches with no host synchronisation
        run()
    torch.cuda.synchronize()
    fresh_status()
    _compare(ref, o)


def test_fp8_and_qkv_chains_same_with_and_without_overlap(C):
    M, H, F = 384, 512, 768
    fi = S.fp8_mlp_inputs(M, H, F, seed=3, with_grad=True)
    h, X, W, Wd, dY = (dev(fi[k]) for k in ("h", "Xq", "Wq", "Wdq", "dY"))
    U8 = torch.uint8
    o = dict(r=torch.empty((M,), device="cuda"), aq=torch.empty((M, F), dtype=U8, device="cuda"),
             am=torch.empty((1,), device="cuda"), Y=torch.empty((M, H), dtype=BF, device="cuda"),
             P=torch.empty((H // 256, M), device="cuda"), Z=torch.empty((M, 2 * F), dtype=BF, device="cuda"),
             dYq=torch.empty((M, H), dtype=U8, device="cuda"), am_dy=torch.empty((1,), device="cuda"),
             eq=torch.empty((M, 2 * F), dtype=U8, device="cuda"), am_e=torch.empty((1,), device="cuda"),
             c=torch.empty((M,), device="cuda"), dh=torch.empty((M, H), dtype=BF, device="cuda"),
             dW_d=torch.empty((H, F), device="cuda"), dW=torch.empty((2 * F, H), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_MLP_FP8_BWD, M, H, F) // 4,), device="cuda")
    qi = S.qkv_inputs(M, H, 768, seed=5)
    hq, Wq, gq = (dev(qi[k]) for k in ("h", "W_qkv", "g"))
    Wqf = torch.empty_like(Wq)
    cos, sin = torch.empty((128, 32), device="cuda"), torch.empty((128, 32), device="cuda")
    o.update(rq=torch.empty((M,), device="cuda"), qkv=torch.empty((M, 768), dtype=BF, device="cuda"))

    def run():
        C.coda_mlp_fp8(h, X, W, Wd, fi["s_x"], fi["s_w"], fi["s_wd"], 0.05, fi["eps"], o["r"], o["aq"], o["am"],
                       o["Y"], o["P"], Z=o["Z"])
        C.coda_mlp_fp8_backward(h, X, W, Wd, o["Z"], o["aq"], o["r"], dY, fi["s_x"], fi["s_w"], fi["s_wd"], 0.05,
                                0.01, 0.002, o["dYq"], o["am_dy"], o["eq"], o["am_e"], o["c"], o["dh"], o["dW_d"],
                                o["dW"], ws)
        C.coda_fold_gain(Wq, gq, Wqf)
        C.coda_rope_table(128, 64, 500000.0, cos, sin)
        C.coda_qkv_rope(hq, Wqf, qi["eps"], 128, 64, 640, cos, sin, o["rq"], o["qkv"])

    C.coda_set_launch_overlap(False)
    run()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in o.items()}
    C.coda_set_launch_overlap(True)
    for v in o.values():
        v.zero_()
    for _ in range(10):
        run()
    torch.cuda.synchronize()
    fresh_status()
    for k in ref:
        if k in ("dW_d", "dW"):
            torch.testing.assert_close(o[k], ref[k], rtol=1e-5, atol=1e-6, msg=k)
        else:
            assert torch.equal(o[k], ref[k]), k


def test_nvfp4_chain_same_with_and_without_overlap(C):
    """The NVFP4 quantiser and MLP chain (whose GEMMs stream their operands early): the same
    codes, scales, amax and Y with the overlap off, on, and issued back to back."""
    M, H, F = 384, 512, 768
    ni = S.nvfp4_mlp_inputs(M, H, F, seed=9, device="cuda")
    sc = lambda t: float(t.abs().max()) / (6 * 448)
    X, W, Wd = C.Nvfp4.empty(M, H, sc(ni["h"])), C.Nvfp4.empty(2 * F, H, sc(ni["W_gu"])), C.Nvfp4.empty(H, F, sc(ni["W_d"]))
    r, amax = torch.empty((M,), device="cuda"), torch.empty((1,), device="cuda")
    a = C.Nvfp4.empty(M, F, 0.01)
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    outs = [X.codes, X.scales, W.codes, W.scales, Wd.codes, Wd.scales, r, a.codes, a.scales, amax, Y, P]

    def run():
        for src, dst in ((ni["W_gu"], W), (ni["W_d"], Wd), (ni["h"], X)):
            C.coda_quantize_nvfp4(src, dst)
        C.coda_mlp_nvfp4(ni["h"], X, W, Wd, 1e-6, r, a, amax, Y, P)

    C.coda_set_launch_overlap(False)
    run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs]
    C.coda_set_launch_overlap(True)
    for t in outs:
        t.zero_()
    for _ in range(10):
        run()
    torch.cuda.synchronize()
    fresh_status()
    for got, want in zip(outs, ref):
        assert torch.equal(got, want)
