"""The block chain captured in a CUDA graph and replayed: the replay gives the same result
as direct calls.  The first call on a device (its set-up: device checks, the tensor-map
encoder, kernel attributes) happens before the capture."""
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
