"""Chains captured in a CUDA graph and replayed (the block forward, the FP8 and NVFP4 MLPs):
the replay gives the same result as direct calls.  The first call on a device (its set-up:
device checks, the tensor-map encoder, kernel attributes) happens before the capture.  And two
chains on two streams at once give the results each gives alone."""
import pytest
import torch

import coda_synth as S
from tests.gpu_helpers import dev, fresh_status

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def test_block_forward_graph_replay_matches_direct_calls():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    C.lib()
    M, H, F = 640, 512, 1024
    inp = S.block_inputs(M, H, F, seed=3)
    d = {k: dev(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    outs = {k: torch.empty(shape, dtype=BF, device="cuda") for k, shape in
            (("h", (M, H)), ("u", (M, H)), ("a", (M, F)), ("Y", (M, H)))}
    r = torch.empty((M,), device="cuda")
    ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")

    def run(stream):
        C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], inp["eps"], outs["h"], r, outs["a"],
                             outs["Y"], ws, g=d["g"], u=outs["u"], stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(s)                         # set-up and a direct result
    torch.cuda.synchronize()
    direct = outs["Y"].clone()
    outs["Y"].zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    fresh_status()
    assert torch.equal(outs["Y"], direct)


def _graph_matches_direct(run, outputs):
    """run(stream) once directly, then captured and replayed: every output equal bit for bit."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(s)
    torch.cuda.synchronize()
    direct = [t.clone() for t in outputs]
    for t in outputs:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    fresh_status()
    for got, want in zip(outputs, direct):
        assert torch.equal(got, want)


def test_fp8_mlp_graph_replay_matches_direct_calls():
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    C.lib()
    M, H, F = 640, 512, 768
    fi = S.fp8_mlp_inputs(M, H, F, seed=5)
    h, X, W, Wd = (dev(fi[k]).contiguous() for k in ("h", "Xq", "Wq", "Wdq"))
    X, W, Wd = (t.view(torch.uint8) for t in (X, W, Wd))
    r = torch.empty((M,), device="cuda")
    aq = torch.empty((M, F), dtype=torch.uint8, device="cuda")
    amax = torch.empty((1,), device="cuda")
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    run = lambda s: C.coda_mlp_fp8(h, X, W, Wd, fi["s_x"], fi["s_w"], fi["s_wd"], 0.05, fi["eps"], r, aq, amax, Y, P,
                                   stream=s)
    _graph_matches_direct(run, [r, aq, amax, Y, P])


def test_nvfp4_mlp_graph_replay_matches_direct_calls():
    """The NVFP4 chain (amax reset, row RMS, two block-scaled GEMMs) has no host step either."""
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    C.lib()
    M, H, F = 640, 512, 768
    ni = S.nvfp4_mlp_inputs(M, H, F, seed=6, device="cuda")
    sc = lambda t: float(t.abs().max()) / (6 * 448)
    X, W, Wd = C.Nvfp4.empty(M, H, sc(ni["h"])), C.Nvfp4.empty(2 * F, H, sc(ni["W_gu"])), C.Nvfp4.empty(H, F, sc(ni["W_d"]))
    for src, dst in ((ni["W_gu"], W), (ni["W_d"], Wd), (ni["h"], X)):
        C.coda_quantize_nvfp4(src, dst)
    r, amax = torch.empty((M,), device="cuda"), torch.empty((1,), device="cuda")
    a = C.Nvfp4.empty(M, F, 0.01)
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    run = lambda s: C.coda_mlp_nvfp4(ni["h"], X, W, Wd, 1e-6, r, a, amax, Y, P, stream=s)
    _graph_matches_direct(run, [r, a.codes, a.scales, amax, Y, P])


def test_two_streams_run_chains_concurrently():
    """Two block-forward chains on two streams at once (their kernels interleave on the GPU):
    each result equals the same chain run alone."""
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    C.lib()
    M, H, F = 640, 512, 1024
    runs = []
    for seed in (7, 8):
        inp = S.block_inputs(M, H, F, seed=seed)
        d = {k: dev(inp[k]) for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
        o = {k: torch.empty(shape, dtype=BF, device="cuda") for k, shape in
             (("h", (M, H)), ("u", (M, H)), ("a", (M, F)), ("Y", (M, H)))}
        o["r"] = torch.empty((M,), device="cuda")
        ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
        runs.append((d, o, ws, inp["eps"]))

    def call(run, stream):
        d, o, ws, eps = run
        C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], eps, o["h"], o["r"], o["a"], o["Y"], ws,
                             g=d["g"], u=o["u"], stream=stream)

    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    alone = []
    for run in runs:
        call(run, s0)
        torch.cuda.synchronize()
        alone.append(run[1]["Y"].clone())
        run[1]["Y"].zero_()
    torch.cuda.synchronize()
    for _ in range(3):                 # interleaved launches on the two streams
        call(runs[0], s0)
        call(runs[1], s1)
    torch.cuda.synchronize()
    fresh_status()
    for run, want in zip(runs, alone):
        assert torch.equal(run[1]["Y"], want)
