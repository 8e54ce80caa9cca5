"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds input generation only: it draws seeded normal samples of the
LLaMA-style shapes and rounds them to the storage dtype with torch's own casts.  It holds
none of the chains' arithmetic, imports neither the oracle nor the CUDA package, and
returns CPU tensors; callers move them to the device.

Recipe (one CPU torch.Generator per call, default seed 0, tensors drawn in the order
listed; N(mu, sigma) uses sigma as the standard deviation):
  tiny fp32 chain:   X, R [M, d] ~ N(0,1); W1 [d, d], W2 [d, n2] ~ N(0, 1/16);
                     g ~ 1 + N(0, 0.1)
  block (1B-shaped): O, R [M, H] ~ N(0,1); W_o [H, H], W_gu [2F, H], W_d [H, F] ~ N(0, w_std);
                     g ~ 1 + N(0, 0.1); dY [M, H] ~ N(0,1)
  qkv:               h [M, H] ~ N(0,1); W_qkv [n_qkv, H] ~ N(0, w_std); g ~ 1 + N(0, 0.1)
  lm head:           h [M, H] ~ N(0,1); g ~ 1 + N(0, 0.1); W_v [V, H] ~ N(0, w_std);
                     targets ~ uniform integers in [0, V) (V = 128256 for LLaMA-3)
  fp8 mlp:           h [M, H] ~ N(0,1); W_gu [2F, H], W_d [H, F] ~ N(0, w_std);
                     e4m3 operands with per-tensor scales amax/448.  The fp8 gate/up
                     weight is taken as the effective weight (any RMSNorm gain already
                     part of it); the workload states no gain for this MLP.
"""
from __future__ import annotations

import torch

E4M3_MAX = 448.0


def _normal(gen, shape, std=1.0, mean=0.0):
    t = torch.empty(shape, dtype=torch.float32, device=gen.device)
    t.normal_(mean=0.0, std=1.0, generator=gen)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def tiny_chain_inputs(M=128, d=256, n2=512, seed=0):
    gen = torch.Generator().manual_seed(seed)
    X = _normal(gen, (M, d))
    R = _normal(gen, (M, d))
    W1 = _normal(gen, (d, d), std=1.0 / 16.0)
    W2 = _normal(gen, (d, n2), std=1.0 / 16.0)
    g = _normal(gen, (d,), std=0.1, mean=1.0)
    return dict(X=X, R=R, W1=W1, W2=W2, g=g, eps=1e-6)


def block_inputs(M, H, F, seed=0, w_std=0.02, with_grad=False, dtype=torch.bfloat16, device="cpu"):
    """device="cuda" draws on the GPU's generator (same recipe, different stream of numbers):
    used where only timing needs the tensors."""
    gen = torch.Generator(device=device).manual_seed(seed)
    out = dict(
        O=_normal(gen, (M, H)).to(dtype),
        R=_normal(gen, (M, H)).to(dtype),
        W_o=_normal(gen, (H, H), std=w_std).to(dtype),
        W_gu=_normal(gen, (2 * F, H), std=w_std).to(dtype),
        W_d=_normal(gen, (H, F), std=w_std).to(dtype),
        g=_normal(gen, (H,), std=0.1, mean=1.0),
        eps=1e-6,
    )
    if with_grad:
        out["dY"] = _normal(gen, (M, H)).to(dtype)
    return out


def qkv_inputs(M, H, n_qkv, seed=0, w_std=0.02, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    return dict(
        h=_normal(gen, (M, H)).to(dtype),
        W_qkv=_normal(gen, (n_qkv, H), std=w_std).to(dtype),
        g=_normal(gen, (H,), std=0.1, mean=1.0),
        eps=1e-6,
    )


def layer_inputs(M, H, F, n_q, n_kv, head_dim, seed=0, w_std=0.02, dtype=torch.bfloat16, device="cpu"):
    """One LLaMA-style decoder layer: input x, attention-input gain g_attn and W_qkv (Q heads,
    then K heads, then V heads), attention-output W_o, MLP gain g_mlp, W_gu (gate rows, then
    up rows) and W_d."""
    gen = torch.Generator(device=device).manual_seed(seed)
    return dict(
        x=_normal(gen, (M, H)).to(dtype),
        g_attn=_normal(gen, (H,), std=0.1, mean=1.0),
        W_qkv=_normal(gen, ((n_q + 2 * n_kv) * head_dim, H), std=w_std).to(dtype),
        W_o=_normal(gen, (H, n_q * head_dim), std=w_std).to(dtype),
        g_mlp=_normal(gen, (H,), std=0.1, mean=1.0),
        W_gu=_normal(gen, (2 * F, H), std=w_std).to(dtype),
        W_d=_normal(gen, (H, F), std=w_std).to(dtype),
        eps=1e-6,
    )


def _to_e4m3(x):
    """Per-tensor e4m3 operand: scale = amax/448, codes = torch's float8_e4m3fn cast of x/scale."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    q = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q, scale


def fp8_mlp_inputs(M, H, F, seed=0, w_std=0.015, with_grad=False):
    gen = torch.Generator().manual_seed(seed)
    h = _normal(gen, (M, H)).to(torch.bfloat16)
    W_gu = _normal(gen, (2 * F, H), std=w_std)
    W_d = _normal(gen, (H, F), std=w_std)
    Xq, s_x = _to_e4m3(h.float())
    Wq, s_w = _to_e4m3(W_gu)
    Wdq, s_wd = _to_e4m3(W_d)
    out = dict(h=h, Xq=Xq, s_x=s_x, Wq=Wq, s_w=s_w, Wdq=Wdq, s_wd=s_wd, eps=1e-6)
    if with_grad:
        out["dY"] = _normal(gen, (M, H)).to(torch.bfloat16)
    return out


def nvfp4_mlp_inputs(M, H, F, seed=0, w_std=0.015, device="cpu"):
    """The FP8 MLP's tensors in bf16 (h ~ N(0, 1), weights ~ N(0, 0.015^2)) for the NVFP4 MLP:
    each side quantises them itself (the library's quantiser on the device, the oracle's on
    the host), with tensor scales amax / (6 * 448)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    h = torch.randn((M, H), generator=gen, device=device).to(torch.bfloat16)
    W_gu = (torch.randn((2 * F, H), generator=gen, device=device) * w_std).to(torch.bfloat16)
    W_d = (torch.randn((H, F), generator=gen, device=device) * w_std).to(torch.bfloat16)
    return dict(h=h, W_gu=W_gu, W_d=W_d, eps=1e-6)


def nvfp4_mlp_bwd_inputs(M, H, F, seed=0, w_std=0.015, device="cpu"):
    """Tensors of the NVFP4 MLP backward in bf16: h ~ N(0, 1), weights ~ N(0, 0.015^2), a saved
    Z = [G | U] ~ N(0, 1), a row scale r ~ 1 + N(0, 0.1^2) (fp32) and an output gradient
    dY ~ N(0, 1); the drawing order is h, W_gu, W_d, Z, r, dY."""
    gen = torch.Generator(device=device).manual_seed(seed)
    bf = torch.bfloat16
    h = torch.randn((M, H), generator=gen, device=device).to(bf)
    W_gu = (torch.randn((2 * F, H), generator=gen, device=device) * w_std).to(bf)
    W_d = (torch.randn((H, F), generator=gen, device=device) * w_std).to(bf)
    Z = torch.randn((M, 2 * F), generator=gen, device=device).to(bf)
    r = 1.0 + 0.1 * torch.randn((M,), generator=gen, device=device)
    dY = torch.randn((M, H), generator=gen, device=device).to(bf)
    return dict(h=h, W_gu=W_gu, W_d=W_d, Z=Z, r=r, dY=dY)


def lm_head_inputs(M, H, V, seed=0, w_std=0.02, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    return dict(
        h=_normal(gen, (M, H)).to(dtype),
        g=_normal(gen, (H,), std=0.1, mean=1.0),
        W_v=_normal(gen, (V, H), std=w_std).to(dtype),
        targets=torch.randint(0, V, (M,), generator=gen, dtype=torch.int32),
        eps=1e-6,
    )
