"""bf16-storage model of the block chains, for tolerances only.

The fp64 oracle is the reference every GPU result is compared with.  This module answers a
different question: how far from the oracle does ANY chain land that stores its
intermediates in bf16 (h, the folded weight W', a, Z, e, dh) and accumulates exactly?
It is the oracle's own arithmetic (same functions, same fused-form order) with a bf16
rounding (torch's cast, round-to-nearest-even) at each point where the chain stores a
tensor.  Its inputs are the same seeded inputs the GPU gets; nothing comes from the GPU.

Tensors that are products of two bf16-rounded GEMM results (a = silu(G) U, e, and the
weight gradients built from them) carry an element-wise error set by that input
rounding, not by the kernels; the parity tests bound the GPU's element-wise error on them
by a small multiple of this model's error on the same elements, besides the 2e-2 normwise
bar."""
import numpy as np
import torch

import oracle as O


def bf(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def block_forward(Oa, R, W_o, g, W_gu, W_d, eps, gain="broadcast"):
    """gain = "broadcast": G1 stores u = bf16(h g) and the gate/up GEMM reads u with the
    unfolded weight; gain = "fold": the gate/up GEMM reads h with W' = bf16(W g)."""
    h = bf(O.linear(Oa, W_o) + R)
    r = f32(1.0 / np.sqrt(np.mean(h * h, axis=1) + eps))
    if gain == "broadcast":
        Wf = W_gu
        Zf = r[:, None] * O.linear(bf(h * g[None, :]), W_gu)
    else:
        Wf = bf(O.fold_gain(W_gu, g))
        Zf = r[:, None] * O.linear(h, Wf)
    F = Zf.shape[1] // 2
    a = bf(O.swiglu(Zf[:, :F], Zf[:, F:]))
    Y = bf(O.linear(a, W_d) + h)
    return dict(h=h, r=r, Z=bf(Zf), a=a, Y=Y, Wf=Wf)


def block_backward(fwd, Oa, W_o, g, W_gu, W_d, dY):
    h, r, Z, a = fwd["h"], fwd["r"], fwd["Z"], fwd["a"]
    H = h.shape[1]
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    dA = dY @ W_d
    e = bf(r[:, None] * np.hstack([dA * U * O.silu_grad(G), dA * O.silu(G)]))
    c = f32(r * np.sum(e * Z, axis=1) / H)
    t = e @ W_gu
    dh = bf(g[None, :] * t - c[:, None] * h + dY)
    return dict(e=e, c=c, dh=dh, dO=bf(dh @ W_o), dW_o=dh.T @ Oa, dW_gu=g[None, :] * (e.T @ h), dW_d=dY.T @ a,
                dg=np.sum(h * t, axis=0))


def normwise(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    m = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / m) if m > 0 else float(np.max(np.abs(got)))
