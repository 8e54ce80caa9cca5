"""Plain fp64 CPU oracle for CODA-style GEMM-epilogue chains.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, links or calls this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
(``cpu_baseline`` and ``--impl reference``) do.  It imports nothing from the CUDA
package either; the two sides share only the seeded input generators in ``coda_synth``.

Sources, by page title and section (the pages print no formulas, only op names; every
function below is the textbook definition of the op the pages name):

* [Ecosistema] "CODA: Nuevo kernel GPU reduce costos de entrenamiento IA"
  (ecosistemastartup.com), section "¿Qué es GEMM-epilogue y por qué importa…?":
  GEMM is C = alpha*A*B + beta*C; the epilogue applies scaling, bias, activation,
  residual addition, precision cast and clamp before the store.
* [KuCoin] "CODA: new research optimizes Transformer training with GEMM-epilogue
  programming" (kucoin.com news flash):
  - "CODA: «El epílogo» esconde un tesoro": in GEMM -> residual -> RMSNorm -> GEMM the
    per-row RMS scale r commutes with the second matmul, so it is applied at the end of
    the second GEMM; the first GEMM only emits partial RMS (partial sums of squares),
    which a very light reduce kernel combines.  The same rewrite covers SwiGLU, RoPE and
    the backward pass.
  - "Cinco «bloques» y un «lenguaje LEGO»": elementwise/pairwise transforms (residual
    add, activation, RoPE), vector load (RMSNorm gain broadcast), matrix-block load/store
    (saved activations), block reduction (local RMS), state change (online max/sum-exp).
  - "hoja de referencia": coverage is RMSNorm, residual add, SwiGLU, RoPE, cross-entropy
    and their gradients, LLaMA-style blocks, everything but attention and embeddings.

Everything is computed in float64 with numpy; ``numpy.matmul`` is the only library
primitive (a GEMM step).  There is no blocking, fusion or reordering beyond what each
definition states.  Two forms are written out for the chains: the plain unfused chain
(normalise, then GEMM; textbook chain rule for backward) and the reparameterised forms
the kernels implement (deferred r, folded gain, fused backward combine); the tests pin
both against each other, against closed forms and against finite differences.

Readings of points the pages leave open (the plainest reading consistent with them):
  1. RMSNorm: r_i = (mean_j h_ij^2 + eps)^(-1/2), eps inside the square root.
  2. "Partial RMS" = partial sums of squares over column tiles (RMS is not additive).
  3. The RMSNorm gain g sits on the next GEMM's K dimension, so the reparameterised form
     folds it into that weight: W'[n, k] = W[n, k] * g[k].
  4. SwiGLU: a = silu(G) * U, gate = rows [0, F) and up = rows [F, 2F) of W_gu.
  5. RoPE pairs adjacent columns (2p, 2p+1) of each head; theta_p = base^(-2p/head_dim);
     position = row index mod sequence length; only the first ``n_rot_cols`` columns
     (the Q and K heads) are rotated.
  6. FP8 is OCP e4m3 ("fn": no infinities, max 448) with round-to-nearest-even and
     saturation to +-448; dequantised value = scale * code value.
  7. Cross-entropy: mean over rows of logsumexp(logits) - logit[target], the final RMSNorm
     before the LM head as in the block chain; every target is a valid class index.
  8. FP8 backward of the MLP: every backward GEMM takes e4m3 operands with per-tensor
     scales like the forward's.  The output gradient dY and the SwiGLU-backward output e
     are quantised with scales the caller supplies (delayed scaling, as for s_a); the GEMMs
     and the row sum behind c see the dequantised values; the residual gradient (+ dY) and
     the RMSNorm-backward combine use dY and h as stored (bf16).
  9. FP4 operands are NVFP4, the block-scaled 4-bit format of the Blackwell tensor cores (the
     pages name FP4 only as a faster matmul format).  Each row of an operand is cut into
     blocks of 16 consecutive K elements.  A block carries one unsigned e4m3 scale sf, the
     tensor carries one fp32 scale s, and an element carries an e2m1 code q (values 0, 0.5,
     1, 1.5, 2, 3, 4, 6 and their negatives); its value is s * sf * q.  Quantising a block is
     the plain definition, in float64: sf = e4m3(amax / (6 s)), then q = e2m1(x / (sf s))
     (zero when sf is zero), both rounded to nearest-even with saturation.  A quantiser that
     takes these steps in fp32 may round the other way where a value lies within an fp32
     rounding of a midpoint; the tests accept exactly those codes.  s is chosen by the
     caller: amax / (6 * 448) of the tensor for operands known up front, and a delayed scale
     (as s_a above) for the SwiGLU output.
 10. NVFP4 backward of the MLP: the block-scaled tensor cores take both operands blocked along
     the GEMM's own K, so every backward GEMM quantises its two operands along its K.  dY is
     quantised along its rows for dA = dY W_d (K = H) and along its columns for dW_d = dY^T a
     (K = tokens); W_d and W_gu are quantised transposed (blocks along F and 2F); e along its
     rows for t = e W_gu (K = 2F) and along its columns for dW = e^T x (K = tokens); a is
     recomputed from the saved Z (a = silu(G) U) and x is the bf16 activation h, both quantised
     along the token axis for the weight gradients.  Scales: s_dy and s_e are the caller's
     delayed scales (as reading 8), s_a the forward's, the others amax / (6 * 448) of their
     tensor.  The row sum behind c uses e before quantisation (the SwiGLU-backward epilogue
     forms it there), and the residual gradient and the combine use dY and h as stored.
Every function here is pinned by a test (closed form, invariant, library special case
or brute force); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(x):
    return np.asarray(x, dtype=F64)


# ---------------------------------------------------------------------------------------
# GEMM  [Ecosistema, "¿Qué es GEMM-epilogue…?"]: C = alpha*A*B + beta*C
# ---------------------------------------------------------------------------------------
def gemm_general(A, B, alpha=1.0, C=None, beta=0.0):
    """C_out = alpha * (A @ B) + beta * C, the GEMM as the page writes it."""
    out = F64(alpha) * (_f64(A) @ _f64(B))
    if C is not None and beta != 0.0:
        out = out + F64(beta) * _f64(C)
    return out


def linear(X, W):
    """Y = X W^T for a weight stored [out, in] (nn.Linear layout): B = W^T above."""
    return gemm_general(X, _f64(W).T)


# ---------------------------------------------------------------------------------------
# RMSNorm and its partial form  [KuCoin, "El epílogo esconde un tesoro"]
# ---------------------------------------------------------------------------------------
def rms_scale(h, eps):
    """Per-row RMSNorm scale r_i = 1 / sqrt(mean_j h_ij^2 + eps)."""
    h = _f64(h)
    return 1.0 / np.sqrt(np.mean(h * h, axis=1) + F64(eps))


def rmsnorm(h, g, eps):
    """y_ij = r_i * h_ij * g_j (RMSNorm with gain g)."""
    h = _f64(h)
    return rms_scale(h, eps)[:, None] * h * _f64(g)[None, :]


def partial_sumsq(h, bn):
    """Per-tile partial sums of squares, layout [ceil(d/bn), M]: P[t, i] = sum_{j in tile t} h_ij^2."""
    h = _f64(h)
    M, d = h.shape
    nparts = (d + bn - 1) // bn
    P = np.zeros((nparts, M), dtype=F64)
    for t in range(nparts):
        blk = h[:, t * bn:(t + 1) * bn]
        P[t] = np.sum(blk * blk, axis=1)
    return P


def rms_scale_from_partials(P, d, eps):
    """The light reduce: r_i = 1 / sqrt(sum_t P[t, i] / d + eps)."""
    return 1.0 / np.sqrt(np.sum(_f64(P), axis=0) / F64(d) + F64(eps))


def fold_gain(W, g):
    """W'[n, k] = W[n, k] * g[k]: the gain moved onto the next GEMM's weight (reading 3)."""
    return _f64(W) * _f64(g)[None, :]


# ---------------------------------------------------------------------------------------
# SwiGLU  [KuCoin, "Cinco bloques…": activation as an elementwise transform]
# ---------------------------------------------------------------------------------------
def sigmoid(x):
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """silu(x) = x / (1 + e^-x)."""
    x = _f64(x)
    return x * sigmoid(x)


def silu_grad(x):
    """d silu / dx = sigma(x) * (1 + x * (1 - sigma(x)))."""
    x = _f64(x)
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


def swiglu(G, U):
    """a = silu(G) * U."""
    return silu(G) * _f64(U)


# ---------------------------------------------------------------------------------------
# RoPE  [KuCoin, "Cinco bloques…": RoPE as a pairwise transform]
# ---------------------------------------------------------------------------------------
def rope_inv_freq(head_dim, base):
    """theta_p = base^(-2p / head_dim), p = 0 .. head_dim/2 - 1."""
    p = np.arange(head_dim // 2, dtype=F64)
    return F64(base) ** (-2.0 * p / F64(head_dim))


def rope_rotate(Z, positions, n_rot_cols, head_dim, base):
    """Rotate each adjacent pair (2p, 2p+1) of every head in columns [0, n_rot_cols) by
    phi = position * theta_p; columns from n_rot_cols on are returned unchanged."""
    Z = _f64(Z)
    out = Z.copy()
    phi = _f64(positions)[:, None] * rope_inv_freq(head_dim, base)[None, :]
    c, s = np.cos(phi), np.sin(phi)
    for h0 in range(0, n_rot_cols, head_dim):
        x0 = Z[:, h0:h0 + head_dim:2]
        x1 = Z[:, h0 + 1:h0 + head_dim:2]
        out[:, h0:h0 + head_dim:2] = x0 * c - x1 * s
        out[:, h0 + 1:h0 + head_dim:2] = x0 * s + x1 * c
    return out


# ---------------------------------------------------------------------------------------
# FP8 e4m3 (reading 6)  [KuCoin, "El impuesto a la pereza": FP8 raises the non-GEMM share]
# ---------------------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_round(x):
    """Nearest e4m3 value, ties to even mantissa, saturating to +-448 (float64 result).

    Normal numbers 2^e * (1 + m/8) with e in [-6, 8]; subnormals m * 2^-9, m in 1..7.
    The spacing at magnitude a is 2^(e-3) with e = max(floor(log2 a), -6)."""
    x = _f64(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.maximum(ex.astype(F64) - 1.0, -6.0)
    q = np.exp2(e - 3.0)
    v = np.rint(a / q) * q                    # numpy rint rounds half to even
    v = np.minimum(v, E4M3_MAX)
    return np.copysign(v, x)


def e4m3_decode(codes):
    """Value of each e4m3 byte: sign | 4-bit exponent (bias 7) | 3-bit mantissa; 0x7f/0xff NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sgn = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = (c & 0x7).astype(F64)
    val = np.where(E == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(E.astype(F64) - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sgn * val


def e4m3_encode(x):
    """e4m3 byte for each value (after e4m3_round): inverse of e4m3_decode on finite codes."""
    v = e4m3_round(x)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1
    normal = a >= 2.0 ** -6
    E = np.where(normal, e + 7, 0)
    M = np.where(normal, np.rint(a / np.exp2(e.astype(F64)) * 8.0 - 8.0), np.rint(a / 2.0 ** -9))
    code = (np.where(sign, 0x80, 0) | (E.astype(np.int64) << 3) | M.astype(np.int64)).astype(np.uint8)
    return code


# ---------------------------------------------------------------------------------------
# NVFP4 (reading 9)  [KuCoin, "El impuesto a la pereza": FP8 and FP4 speed up the matmul,
# so the tensor traffic around it weighs more]
# ---------------------------------------------------------------------------------------
E2M1_MAX = 6.0
NVFP4_BLOCK = 16


def e2m1_round(x):
    """Nearest e2m1 value, ties to the even code, saturating to +-6 (float64 result).

    e2m1 = sign | 2-bit exponent (bias 1) | 1-bit mantissa: subnormals 0 and 0.5, then
    1, 1.5, 2, 3, 4, 6.  The spacing at magnitude a is 2^(e-1) with e = max(floor(log2 a), 0),
    and an even multiple of the spacing is an even code."""
    x = _f64(x)
    a = np.minimum(np.abs(x), E2M1_MAX)
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(F64) - 1.0, 0.0)
    q = np.exp2(e - 1.0)
    v = np.minimum(np.rint(a / q) * q, E2M1_MAX)
    return np.copysign(v, x)


def e2m1_decode(codes):
    """Value of each 4-bit code (low nibble of the input): sign bit 3, exponent bits 2-1, mantissa bit 0."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sgn = np.where(c & 0x8, -1.0, 1.0)
    E = (c >> 1) & 0x3
    m = (c & 0x1).astype(F64)
    val = np.where(E == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(E.astype(F64) - 1.0))
    return sgn * val


def e2m1_encode(x):
    """4-bit code of each value (after e2m1_round): inverse of e2m1_decode; -0 keeps its sign bit."""
    v = e2m1_round(x)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1
    normal = a >= 1.0
    E = np.where(normal, e + 1, 0)
    M = np.where(normal, np.rint(a / np.exp2(e.astype(F64)) * 2.0 - 2.0), np.rint(a * 2.0))
    return (np.where(sign, 0x8, 0) | (E.astype(np.int64) << 1) | M.astype(np.int64)).astype(np.uint8)


def nvfp4_quantize(x, s):
    """NVFP4 quantisation of x [R, K] (K a multiple of 16) with the tensor scale s (reading 9).

    Returns (q, sf): q [R, K] e2m1 values and sf [R, K / 16] e4m3 block scales (float64), so
    that the dequantised tensor is s * sf (repeated over each block) * q.  Every step is the
    float64 definition: sf = e4m3(amax / (6 s)), q = e2m1(x / (sf s)), q = 0 where sf = 0."""
    x = _f64(x)
    R, K = x.shape
    assert K % NVFP4_BLOCK == 0
    xb = x.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    amax = np.max(np.abs(xb), axis=2)
    sf = e4m3_round(amax / (E2M1_MAX * F64(s)))
    d = (sf * F64(s))[:, :, None]
    y = np.where(d > 0, xb / np.where(d > 0, d, 1.0), 0.0)
    q = e2m1_round(y).reshape(R, K)
    return q, sf


def nvfp4_dequantize(q, sf, s):
    """s * sf * q with each block scale spread over its 16 elements."""
    q, sf = _f64(q), _f64(sf)
    return F64(s) * np.repeat(sf, NVFP4_BLOCK, axis=1) * q


def nvfp4_round_rows(x, s):
    """x [R, K] quantised along its rows (blocks of 16 consecutive columns) and dequantised."""
    q, sf = nvfp4_quantize(x, s)
    return nvfp4_dequantize(q, sf, s)


def nvfp4_round_cols(x, s):
    """x [R, K] quantised along its columns (blocks of 16 consecutive rows) and dequantised:
    the row quantisation of the transpose, transposed back."""
    return nvfp4_round_rows(_f64(x).T, s).T


def mlp_nvfp4(h, Xq, Xsf, s_x, Wq, Wsf, s_w, Wdq, Wdsf, s_wd, s_a, eps, bn):
    """The FP8 MLP above with NVFP4 operands (reading 9).  x, W (the effective gate/up weight)
    and W_d are given as (codes, block scales, tensor scale); r comes from the bf16 h.
      Z = r * (x W^T);  a = silu(G) U;  amax = max |a|;  (a_q, a_sf) = nvfp4(a, s_a);
      Y = nvfp4_dequantize(a_q, a_sf, s_a) W_d^T + h;  P = partial sums of squares of Y."""
    r = rms_scale(h, eps)
    Z = r[:, None] * linear(nvfp4_dequantize(Xq, Xsf, s_x), nvfp4_dequantize(Wq, Wsf, s_w))
    F = Z.shape[1] // 2
    a = swiglu(Z[:, :F], Z[:, F:])
    aq, asf = nvfp4_quantize(a, s_a)
    Y = linear(nvfp4_dequantize(aq, asf, s_a), nvfp4_dequantize(Wdq, Wdsf, s_wd)) + _f64(h)
    return dict(r=r, Z=Z, a=a, amax=float(np.max(np.abs(a))), aq=aq, asf=asf, Y=Y, P=partial_sumsq(Y, bn))


# ---------------------------------------------------------------------------------------
# Chains.  Plain (unfused) forms first, then the reparameterised forms the kernels use.
# ---------------------------------------------------------------------------------------
def tiny_chain(X, R, W1, W2, g, eps):
    """Tiny GEMM -> residual -> RMSNorm -> GEMM, weights in [in, out] form:
    out = rmsnorm(X W1 + R, g) W2."""
    h = gemm_general(X, W1) + _f64(R)
    return dict(h=h, r=rms_scale(h, eps), out=gemm_general(rmsnorm(h, g, eps), W2))


def block_forward(O, R, W_o, g, W_gu, W_d, eps):
    """LLaMA-style block tail, plain unfused chain (weights [out, in]):
    h = O W_o^T + R;  y = rmsnorm(h, g);  Z = y W_gu^T = [G | U];  a = silu(G) U;
    Y = a W_d^T + h."""
    h = linear(O, W_o) + _f64(R)
    r = rms_scale(h, eps)
    y = r[:, None] * h * _f64(g)[None, :]
    Z = linear(y, W_gu)
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    a = swiglu(G, U)
    Y = linear(a, W_d) + h
    return dict(h=h, r=r, y=y, Z=Z, G=G, U=U, a=a, Y=Y)


def block_forward_deferred(O, R, W_o, g, W_gu, W_d, eps, bn):
    """The reparameterised chain [KuCoin, "El epílogo esconde un tesoro"]: GEMM1 emits
    partial sums of squares, a light reduce turns them into r, and r is applied per row
    after the second GEMM, whose weight carries the folded gain."""
    h = linear(O, W_o) + _f64(R)
    P = partial_sumsq(h, bn)
    r = rms_scale_from_partials(P, h.shape[1], eps)
    Z = r[:, None] * linear(h, fold_gain(W_gu, g))
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    a = swiglu(G, U)
    Y = linear(a, W_d) + h
    return dict(h=h, P=P, r=r, Z=Z, G=G, U=U, a=a, Y=Y)


def block_backward(fwd, O, W_o, g, W_gu, W_d, dY):
    """Plain chain rule through the unfused ops of ``block_forward`` (RMSNorm backward in
    its textbook form dh = r (g*dy) - (r^3/d) h sum_j g_j dy_j h_j)."""
    h, r, y, G, U, a = (fwd[k] for k in ("h", "r", "y", "G", "U", "a"))
    dY = _f64(dY)
    W_d, W_gu, W_o, g = _f64(W_d), _f64(W_gu), _f64(W_o), _f64(g)
    d = h.shape[1]
    dW_d = dY.T @ a
    da = dY @ W_d
    dG = da * U * silu_grad(G)
    dU = da * silu(G)
    dZ = np.hstack([dG, dU])
    dW_gu = dZ.T @ y
    dy = dZ @ W_gu
    dg = np.sum(dy * r[:, None] * h, axis=0)
    proj = np.sum(g[None, :] * dy * h, axis=1)
    dh = r[:, None] * (g[None, :] * dy) - (r ** 3 / d)[:, None] * h * proj[:, None] + dY
    dO = dh @ W_o
    dW_o = dh.T @ _f64(O)
    return dict(dW_d=dW_d, da=da, dZ=dZ, dW_gu=dW_gu, dg=dg, dh=dh, dR=dh, dO=dO, dW_o=dW_o)


def block_backward_fused(fwd, O, W_o, g, W_gu, W_d, dY):
    """The fused backward forms the kernels compute (each GEMM + its epilogue):
      e   = r * [dG | dU]          (SwiGLU-backward epilogue on dA = dY W_d, row scale r)
      s_i = sum_k e_ik Z_ik        (row dot partial), c_i = r_i s_i / d (light reduce)
      t   = e W_gu;  dh = g*t - c*h + dY;  dg_j = sum_i h_ij t_ij   (RMSNorm-bwd combine)
      dW_gu[n, k] = g_k (e^T h)[n, k];  dW_d = dY^T a;  dO = dh W_o;  dW_o = dh^T O."""
    h, r, Z, G, U, a = (fwd[k] for k in ("h", "r", "Z", "G", "U", "a"))
    dY = _f64(dY)
    W_d, W_gu, W_o, g = _f64(W_d), _f64(W_gu), _f64(W_o), _f64(g)
    d = h.shape[1]
    dA = dY @ W_d
    e = r[:, None] * np.hstack([dA * U * silu_grad(G), dA * silu(G)])
    s = np.sum(e * Z, axis=1)
    c = r * s / d
    t = e @ W_gu
    dh = g[None, :] * t - c[:, None] * h + dY
    dg = np.sum(h * t, axis=0)
    dW_gu = g[None, :] * (e.T @ h)
    dW_d = dY.T @ a
    dO = dh @ W_o
    dW_o = dh.T @ _f64(O)
    return dict(e=e, s=s, c=c, t=t, dh=dh, dR=dh, dg=dg, dW_gu=dW_gu, dW_d=dW_d, dO=dO, dW_o=dW_o)


def qkv_rope(h, g, W_qkv, eps, seq_len, n_rot_cols, head_dim, base):
    """Input RMSNorm -> QKV projection -> RoPE on the Q and K columns (plain chain)."""
    y = rmsnorm(h, g, eps)
    Z = linear(y, W_qkv)
    pos = np.arange(Z.shape[0]) % seq_len
    return dict(r=rms_scale(h, eps), Z=Z, out=rope_rotate(Z, pos, n_rot_cols, head_dim, base))


def qkv_rope_backward(h, g, W_qkv, dout, eps, seq_len, n_rot_cols, head_dim, base):
    """Plain chain rule through qkv_rope (RMSNorm -> QKV GEMM -> RoPE) for an upstream
    gradient dout of its output: dZ = RoPE^T dout (rotation by -phi); dW = dZ^T y;
    dy = dZ W; RMSNorm backward in its textbook form -> dh, dg."""
    h, g, W = _f64(h), _f64(g), _f64(W_qkv)
    M, d = h.shape
    r = rms_scale(h, eps)
    y = r[:, None] * h * g[None, :]
    pos = np.arange(M) % seq_len
    dZ = rope_rotate(dout, -pos, n_rot_cols, head_dim, base)
    dy = dZ @ W
    dg = np.sum(dy * r[:, None] * h, axis=0)
    proj = np.sum(g[None, :] * dy * h, axis=1)
    dh = r[:, None] * (g[None, :] * dy) - (r ** 3 / d)[:, None] * h * proj[:, None]
    return dict(dZ=dZ, dW=dZ.T @ y, dh=dh, dg=dg)


def qkv_rope_backward_fused(h, g, W_qkv, dout, out, eps, seq_len, n_rot_cols, head_dim, base):
    """The fused forms: e = r RoPE^T(dout) (row-wise pass); s_i = sum_n e_in Z_in, which equals
    r_i sum_n dout_in out_in because the rotation keeps inner products; c = r s / d;
    t = e W;  dh = g t - c h;  dg = sum_rows h t;  dW[n, k] = g_k (e^T h)[n, k]."""
    h, g, W = _f64(h), _f64(g), _f64(W_qkv)
    M, d = h.shape
    r = rms_scale(h, eps)
    pos = np.arange(M) % seq_len
    e = r[:, None] * rope_rotate(dout, -pos, n_rot_cols, head_dim, base)
    s = r * np.sum(_f64(dout) * _f64(out), axis=1)
    c = r * s / d
    t = e @ W
    return dict(e=e, c=c, dh=g[None, :] * t - c[:, None] * h, dg=np.sum(h * t, axis=0),
                dW=g[None, :] * (e.T @ h))


def mlp_fp8(h, Xq_val, s_x, Wq_val, s_w, Wdq_val, s_wd, s_a, eps, bn):
    """FP8 MLP with per-tensor scales.  Operands are e4m3 code values (already decoded to
    float64) with fp32 scales: x = s_x Xq, W = s_w Wq (the effective gate/up weight),
    W_d = s_wd Wdq.  r comes from the bf16 activation h.
      Z = r * (x W'^T);  a = silu(G) U;  amax = max |a|;  a_q = e4m3(a / s_a);
      Y = (s_a a_q) W_d^T + h;  P = partial sums of squares of Y."""
    r = rms_scale(h, eps)
    Z = r[:, None] * linear(F64(s_x) * _f64(Xq_val), F64(s_w) * _f64(Wq_val))
    F = Z.shape[1] // 2
    a = swiglu(Z[:, :F], Z[:, F:])
    aq_val = e4m3_round(a / F64(s_a))
    Y = linear(F64(s_a) * aq_val, F64(s_wd) * _f64(Wdq_val)) + _f64(h)
    return dict(r=r, Z=Z, a=a, amax=np.max(np.abs(a)), aq_val=aq_val, Y=Y, P=partial_sumsq(Y, bn))


def mlp_fp8_backward(h, Xq_val, s_x, Wq_val, s_w, Wdq_val, s_wd, Z, aq_val, s_a, r, dY, s_dy, s_e,
                     quant=e4m3_round):
    """Backward of mlp_fp8 with e4m3 GEMM operands (reading 8).  Saved from the forward: Z =
    [G | U] (post-r, pre-activation), a_q and r.  W = s_w Wq, W_d = s_wd Wdq, x = s_x Xq.
      dY_q = quant(dY / s_dy);  dA = (s_dy dY_q) W_d
      e = r [dA U silu'(G) | dA silu(G)];  e_q = quant(e / s_e);  e_hat = s_e e_q
      c_i = r_i sum_k e_hat_ik Z_ik / H          (RMSNorm backward, scale-invariant part)
      t = e_hat W;  dh = t - c h + dY
      dW_d = (s_dy dY_q)^T (s_a a_q);  dW = e_hat^T x
    ``quant`` is the quantiser (identity gives the exact-arithmetic chain rule)."""
    h, Z, r, dY = _f64(h), _f64(Z), _f64(r), _f64(dY)
    x = F64(s_x) * _f64(Xq_val)
    W = F64(s_w) * _f64(Wq_val)
    W_d = F64(s_wd) * _f64(Wdq_val)
    a = F64(s_a) * _f64(aq_val)
    H = h.shape[1]
    F = Z.shape[1] // 2
    dYq_val = quant(dY / F64(s_dy))
    dYd = F64(s_dy) * dYq_val
    dA = dYd @ W_d
    G, U = Z[:, :F], Z[:, F:]
    e = r[:, None] * np.hstack([dA * U * silu_grad(G), dA * silu(G)])
    eq_val = quant(e / F64(s_e))
    e_hat = F64(s_e) * eq_val
    s = np.sum(e_hat * Z, axis=1)
    c = r * s / H
    t = e_hat @ W
    dh = t - c[:, None] * h + dY
    return dict(dYq_val=dYq_val, amax_dy=float(np.max(np.abs(dY))), dA=dA, e=e, eq_val=eq_val,
                amax_e=float(np.max(np.abs(e))), e_hat=e_hat, s=s, c=c, t=t, dh=dh, dW_d=dYd.T @ a,
                dW=e_hat.T @ x)


def mlp_nvfp4_backward(h, W_gu, W_d, Z, r, dY, s_dy, s_e, s_a, s_x, s_wt, s_wdt, quant=True, round_rows=None,
                       round_cols=None):
    """Backward of the MLP with NVFP4 GEMM operands (reading 10).  h, W_gu (the effective
    gate/up weight, [2F, H]), W_d ([H, F]) and dY are the bf16 tensors; Z = [G | U] and r are
    saved by the forward.  Rr / Rc quantise along rows / columns: nvfp4_round_rows / _cols, or
    the caller's round_rows / round_cols (a test that takes the rounding decisions in another
    precision), or the identity when quant is False:
      dA = Rr(dY, s_dy) Rr(W_d^T, s_wdt)^T;  e = r [dA U silu'(G) | dA silu(G)]
      s_i = sum_k e_ik Z_ik;  c = r s / H
      t = Rr(e, s_e) Rr(W_gu^T, s_wt)^T;  dh = t - c h + dY
      dW_d = Rc(dY, s_dy)^T Rc(silu(G) U, s_a);  dW = Rc(e, s_e)^T Rc(h, s_x)"""
    h, W_gu, W_d, Z, r, dY = (_f64(v) for v in (h, W_gu, W_d, Z, r, dY))
    Rr = (round_rows or nvfp4_round_rows) if quant else (lambda x, s: _f64(x))
    Rc = (round_cols or nvfp4_round_cols) if quant else (lambda x, s: _f64(x))
    H = h.shape[1]
    F = Z.shape[1] // 2
    G, U = Z[:, :F], Z[:, F:]
    dA = Rr(dY, s_dy) @ Rr(W_d.T, s_wdt).T
    e = r[:, None] * np.hstack([dA * U * silu_grad(G), dA * silu(G)])
    s = np.sum(e * Z, axis=1)
    c = r * s / H
    t = Rr(e, s_e) @ Rr(W_gu.T, s_wt).T
    dh = t - c[:, None] * h + dY
    a = swiglu(G, U)
    dW_d = Rc(dY, s_dy).T @ Rc(a, s_a)
    dW = Rc(e, s_e).T @ Rc(h, s_x)
    return dict(dA=dA, e=e, amax_e=float(np.max(np.abs(e))), amax_dy=float(np.max(np.abs(dY))), s=s, c=c, t=t,
                dh=dh, a=a, dW_d=dW_d, dW=dW)


# ---------------------------------------------------------------------------------------
# Cross-entropy after the final RMSNorm and the LM-head GEMM
# [KuCoin, "Cinco bloques…": block log-sum-exp, and max / sum-exp statistics for online
# normalisation; "hoja de referencia": cross-entropy and its gradient are covered]
# ---------------------------------------------------------------------------------------
def logsumexp(z):
    """Row-wise log(sum_j exp(z_ij)), shifted by the row maximum (exact in real arithmetic)."""
    z = _f64(z)
    m = np.max(z, axis=1)
    return m + np.log(np.sum(np.exp(z - m[:, None]), axis=1))


def cross_entropy(logits, targets):
    """Per-row loss_i = logsumexp(logits_i) - logits_i[target_i], and their mean."""
    z = _f64(logits)
    t = np.asarray(targets, dtype=np.int64)
    lse = logsumexp(z)
    loss = lse - z[np.arange(z.shape[0]), t]
    return dict(lse=lse, loss=loss, mean=float(np.mean(loss)))


def lm_head_xent_forward(h, g, W_v, targets, eps):
    """Final RMSNorm, LM head and mean cross-entropy (plain chain):
    y = rmsnorm(h, g);  logits = y W_v^T;  loss = mean_i (lse_i - logits_i[t_i])."""
    r = rms_scale(h, eps)
    y = r[:, None] * _f64(h) * _f64(g)[None, :]
    logits = linear(y, W_v)
    ce = cross_entropy(logits, targets)
    return dict(r=r, y=y, logits=logits, **ce)


def lm_head_xent_backward(fwd, h, g, W_v, targets, dloss=1.0):
    """Plain chain rule of lm_head_xent_forward for an upstream gradient dloss of the mean:
    dlogits = dloss (softmax(logits) - onehot(t)) / M;  dW_v = dlogits^T y;  dy = dlogits W_v;
    RMSNorm backward (textbook form) -> dh, dg."""
    logits, r, y = fwd["logits"], fwd["r"], fwd["y"]
    h, g, W_v = _f64(h), _f64(g), _f64(W_v)
    M, d = h.shape
    p = np.exp(logits - fwd["lse"][:, None])
    onehot = np.zeros_like(p)
    onehot[np.arange(M), np.asarray(targets, dtype=np.int64)] = 1.0
    dlogits = F64(dloss) * (p - onehot) / F64(M)
    dW_v = dlogits.T @ y
    dy = dlogits @ W_v
    dg = np.sum(dy * r[:, None] * h, axis=0)
    proj = np.sum(g[None, :] * dy * h, axis=1)
    dh = r[:, None] * (g[None, :] * dy) - (r ** 3 / d)[:, None] * h * proj[:, None]
    return dict(dlogits=dlogits, dW_v=dW_v, dh=dh, dg=dg)


def lm_head_xent_backward_fused(fwd, h, g, W_v, targets, dloss=1.0):
    """The fused forms the kernels compute:
      e = r * dloss (exp(z - lse) - onehot) / M   with z = logits (softmax-gradient epilogue)
      s_i = sum_v e_iv z_iv,  c = r s / d;  t = e W_v;  dh = g t - c h;  dg = sum_i h t
      dW_v = e^T u with u = h g."""
    logits, r = fwd["logits"], fwd["r"]
    h, g, W_v = _f64(h), _f64(g), _f64(W_v)
    M, d = h.shape
    onehot = np.zeros_like(logits)
    onehot[np.arange(M), np.asarray(targets, dtype=np.int64)] = 1.0
    e = r[:, None] * F64(dloss) * (np.exp(logits - fwd["lse"][:, None]) - onehot) / F64(M)
    s = np.sum(e * logits, axis=1)
    c = r * s / d
    t = e @ W_v
    dh = g[None, :] * t - c[:, None] * h
    return dict(e=e, c=c, dh=dh, dg=np.sum(h * t, axis=0), dW_v=e.T @ (h * g[None, :]))


def xent_partials(z, bn):
    """Per-tile online-normalisation state of each row: for tile t of bn columns,
    m[t, i] = max_j z_ij and s[t, i] = sum_j exp(z_ij - m[t, i]) (layout [ntiles, M])."""
    z = _f64(z)
    M, V = z.shape
    n = (V + bn - 1) // bn
    m = np.zeros((n, M))
    s = np.zeros((n, M))
    for t in range(n):
        blk = z[:, t * bn:(t + 1) * bn]
        m[t] = np.max(blk, axis=1)
        s[t] = np.sum(np.exp(blk - m[t][:, None]), axis=1)
    return m, s


def xent_combine(m, s):
    """The light reduce of the partial states: lse = M + log(sum_t s_t exp(m_t - M)),
    M = max_t m_t."""
    m, s = _f64(m), _f64(s)
    top = np.max(m, axis=0)
    return top + np.log(np.sum(s * np.exp(m - top[None, :]), axis=0))


# ---------------------------------------------------------------------------------------
# Error metric used by every parity test
# ---------------------------------------------------------------------------------------
def max_rel_err(got, ref):
    """max_i |got_i - ref_i| / max(|ref_i|, rms(ref)): relative error with an RMS floor so
    that entries near zero do not dominate."""
    got, ref = _f64(got), _f64(ref)
    floor = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    den = np.maximum(np.abs(ref), floor)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(got - ref) / den)) if ref.size else 0.0
