"""ctypes binding of libcoda.so (include/coda.h): argument marshalling only.

Every function here turns torch tensors (device memory owned by the caller) into the
plain pointers, sizes and layouts of the C ABI and calls the library; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the library is
not built or cannot be loaded, loading raises CodaLibraryError, and a non-zero status
from a call raises CodaError.

A 2-D tensor's layout is read from its strides: stride (ld, 1) is CODA_ROW_MAJOR with
leading dimension ld; stride (1, ld) is CODA_COL_MAJOR (a transposed view, e.g. x.t()).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_uint32, c_void_p

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libcoda.so")

# ----------------------------------------------------------------------- constants
OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_UNSUPPORTED_PROGRAM, ERR_LAUNCH, ERR_DEVICE_TIMEOUT, ERR_NO_DEVICE = (
    0, -1, -2, -3, -4, -5, -6, -7, -8)
F32, BF16, E4M3, NVFP4 = 0, 1, 2, 3
ROW_MAJOR, COL_MAJOR = 0, 1
OP_TENSOR_SCALE, OP_ROW_SCALE, OP_COL_SCALE, OP_ADD_SIDE, OP_SWIGLU, OP_ROPE = 1, 2, 3, 4, 5, 6
OP_SWIGLU_BWD, OP_RMSBWD_COMBINE, OP_ROW_SUMSQ_PARTIAL, OP_ROW_DOT_PARTIAL = 7, 8, 9, 10
OP_COL_DOT_PARTIAL, OP_AMAX, OP_STORE_AUX, OP_STORE_COL_SCALED, OP_XENT_PARTIAL, OP_XENT_BWD = 11, 12, 13, 14, 15, 16
REDUCE_RSQRT_MEAN, REDUCE_SCALE_SUM = 0, 1
WS_BLOCK_FWD, WS_BLOCK_BWD, WS_XENT_FWD, WS_XENT_BWD, WS_MLP_FP8_BWD, WS_MLP_NVFP4_BWD = 0, 1, 2, 3, 4, 5
MAX_OPS = 8

EXPORTED = [
    "coda_gemm_epilogue", "coda_rms_partial_reduce", "coda_row_rms", "coda_col_reduce", "coda_fold_gain",
    "coda_rope_table", "coda_block_forward", "coda_block_backward", "coda_qkv_rope", "coda_mlp_fp8",
    "coda_workspace_size", "coda_get_device_status", "coda_set_watchdog_ms", "coda_inject_dropped_stage",
    "coda_device_sm_count", "coda_status_string", "coda_version", "coda_block_forward_noalloc", "coda_rms_gain",
    "coda_xent_combine", "coda_lm_head_xent_forward", "coda_lm_head_xent_backward", "coda_rope_backward",
    "coda_qkv_rope_backward", "coda_mlp_fp8_backward", "coda_quantize_e4m3", "coda_set_launch_overlap",
    "coda_quantize_nvfp4", "coda_nvfp4_scale_bytes", "coda_mlp_nvfp4", "coda_quantize_nvfp4_t",
    "coda_mlp_nvfp4_backward",
]
NOALLOC_MAX_PARTIALS = 1 << 20


class CodaLibraryError(RuntimeError):
    pass


class CodaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


# ---------------------------------------------------------------------- structures
class CodaTensor(Structure):
    _fields_ = [("ptr", c_void_p), ("dtype", c_int32), ("layout", c_int32), ("rows", c_int64), ("cols", c_int64),
                ("ld", c_int64)]


class CodaProgram(Structure):
    _fields_ = [("n_ops", c_int32), ("ops", c_int32 * MAX_OPS)]


class CodaSide(Structure):
    _fields_ = [("residual", POINTER(CodaTensor)), ("row_scale", c_void_p), ("row_coef", c_void_p),
                ("col_scale", c_void_p), ("aux_in", POINTER(CodaTensor)), ("aux_in2", POINTER(CodaTensor)),
                ("rope_cos", c_void_p), ("rope_sin", c_void_p), ("rope_seq_len", c_int32),
                ("rope_head_dim", c_int32), ("rope_ncols", c_int32), ("tensor_scale", c_float),
                ("out_scale", c_float), ("row_index", c_void_p), ("a_block_scales", c_void_p),
                ("w_block_scales", c_void_p), ("out_fp4_scale", c_float)]


class CodaAux(Structure):
    _fields_ = [("row_partials", c_void_p), ("row_partials_ld", c_int64), ("col_partials", c_void_p),
                ("col_partials_ld", c_int64), ("store_aux", POINTER(CodaTensor)), ("amax", c_void_p),
                ("row_partials2", c_void_p), ("row_values", c_void_p), ("out_block_scales", c_void_p)]


class CodaBlockFwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("eps", c_float), ("O", c_void_p), ("R", c_void_p),
                ("W_o", c_void_p), ("W_gu", c_void_p), ("W_d", c_void_p), ("g", c_void_p), ("u", c_void_p),
                ("h", c_void_p), ("r", c_void_p), ("a", c_void_p), ("Y", c_void_p), ("Z", c_void_p),
                ("Y_partials", c_void_p), ("workspace", c_void_p)]


class CodaBlockBwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("O", c_void_p), ("W_o", c_void_p),
                ("W_gu", c_void_p), ("W_d", c_void_p), ("g", c_void_p), ("h", c_void_p), ("r", c_void_p),
                ("Z", c_void_p), ("a", c_void_p), ("dY", c_void_p), ("e", c_void_p), ("dh", c_void_p),
                ("dO", c_void_p), ("dW_o", c_void_p), ("dW_gu", c_void_p), ("dW_d", c_void_p), ("dg", c_void_p),
                ("c", c_void_p), ("workspace", c_void_p)]


class CodaQkvRope(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("N", c_int64), ("seq_len", c_int32), ("head_dim", c_int32),
                ("rope_ncols", c_int32), ("eps", c_float), ("h", c_void_p), ("W_qkv", c_void_p),
                ("rope_cos", c_void_p), ("rope_sin", c_void_p), ("r", c_void_p), ("out", c_void_p)]


class CodaMlpFp8(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("eps", c_float), ("s_x", c_float),
                ("s_w", c_float), ("s_wd", c_float), ("s_a", c_float), ("h", c_void_p), ("X_q", c_void_p),
                ("W_q", c_void_p), ("W_dq", c_void_p), ("r", c_void_p), ("a_q", c_void_p), ("amax", c_void_p),
                ("Y", c_void_p), ("Y_partials", c_void_p), ("Z", c_void_p)]


class CodaMlpNvfp4(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("eps", c_float), ("s_x", c_float),
                ("s_w", c_float), ("s_wd", c_float), ("s_a", c_float), ("h", c_void_p), ("X_q", c_void_p),
                ("X_sf", c_void_p), ("W_q", c_void_p), ("W_sf", c_void_p), ("W_dq", c_void_p), ("W_dsf", c_void_p),
                ("r", c_void_p), ("a_q", c_void_p), ("a_sf", c_void_p), ("amax", c_void_p), ("Y", c_void_p),
                ("Y_partials", c_void_p)]


class CodaMlpNvfp4Bwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("s_x", c_float), ("s_wt", c_float),
                ("s_wdt", c_float), ("s_a", c_float), ("s_dy", c_float), ("s_e", c_float)] + \
               [(n, c_void_p) for n in ("h", "W_guT", "W_guT_sf", "W_dT", "W_dT_sf", "Z", "r", "dY", "dY_r", "dY_r_sf",
                                        "dY_c", "dY_c_sf", "e", "e_r", "e_r_sf", "e_c", "e_c_sf", "a_c", "a_c_sf",
                                        "x_c", "x_c_sf", "amax_dy", "amax_e", "c", "dh", "dW_d", "dW", "workspace")]


class CodaMlpFp8Bwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("F", c_int64), ("s_x", c_float), ("s_w", c_float),
                ("s_wd", c_float), ("s_a", c_float), ("s_dy", c_float), ("s_e", c_float), ("h", c_void_p),
                ("X_q", c_void_p), ("W_q", c_void_p), ("W_dq", c_void_p), ("Z", c_void_p), ("a_q", c_void_p),
                ("r", c_void_p), ("dY", c_void_p), ("dY_q", c_void_p), ("amax_dy", c_void_p), ("e_q", c_void_p),
                ("amax_e", c_void_p), ("c", c_void_p), ("dh", c_void_p), ("dW_d", c_void_p), ("dW", c_void_p),
                ("workspace", c_void_p)]


class CodaXentFwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("V", c_int64), ("eps", c_float), ("h", c_void_p), ("g", c_void_p),
                ("W_v", c_void_p), ("targets", c_void_p), ("u", c_void_p), ("r", c_void_p), ("lse", c_void_p),
                ("loss", c_void_p), ("loss_mean", c_void_p), ("workspace", c_void_p)]


class CodaXentBwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("V", c_int64), ("dloss", c_float), ("h", c_void_p),
                ("g", c_void_p), ("W_v", c_void_p), ("targets", c_void_p), ("u", c_void_p), ("r", c_void_p),
                ("lse", c_void_p), ("e", c_void_p), ("dh", c_void_p), ("dW_v", c_void_p), ("dg", c_void_p),
                ("c", c_void_p), ("workspace", c_void_p)]


class CodaQkvRopeBwd(Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("N", c_int64), ("seq_len", c_int32), ("head_dim", c_int32),
                ("rope_ncols", c_int32), ("h", c_void_p), ("g", c_void_p), ("W_qkv", c_void_p), ("r", c_void_p),
                ("out", c_void_p), ("dout", c_void_p), ("dres", c_void_p), ("rope_cos", c_void_p),
                ("rope_sin", c_void_p), ("e", c_void_p), ("dh", c_void_p), ("dW_qkv", c_void_p), ("dg", c_void_p),
                ("c", c_void_p), ("workspace", c_void_p)]


# --------------------------------------------------------------------- the library
_lib = None


def lib():
    """The loaded libcoda.so (raises CodaLibraryError if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise CodaLibraryError(f"libcoda.so is not built ({LIB_PATH}); run __graft_entry__.build() or "
                               "python -m gemm_epilogue_transformer_tcgen05_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    P = POINTER
    sigs = {
        "coda_gemm_epilogue": [P(CodaTensor), P(CodaTensor), P(CodaProgram), P(CodaSide), P(CodaTensor), P(CodaAux),
                               c_void_p],
        "coda_rms_partial_reduce": [c_void_p, c_int64, c_int32, c_int64, c_int64, c_float, c_int32, c_void_p, c_void_p,
                                    c_void_p],
        "coda_row_rms": [P(CodaTensor), c_float, c_void_p, c_void_p],
        "coda_col_reduce": [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p],
        "coda_fold_gain": [P(CodaTensor), c_void_p, c_float, P(CodaTensor), c_void_p],
        "coda_rope_table": [c_int32, c_int32, c_double, c_void_p, c_void_p, c_void_p],
        "coda_block_forward": [P(CodaBlockFwd), c_void_p],
        "coda_block_forward_noalloc": [P(CodaBlockFwd), c_void_p],
        "coda_block_backward": [P(CodaBlockBwd), c_void_p],
        "coda_qkv_rope": [P(CodaQkvRope), c_void_p],
        "coda_mlp_fp8": [P(CodaMlpFp8), c_void_p],
        "coda_mlp_fp8_backward": [P(CodaMlpFp8Bwd), c_void_p],
        "coda_quantize_e4m3": [P(CodaTensor), c_float, P(CodaTensor), c_void_p, c_void_p],
        "coda_get_device_status": [c_void_p, P(c_int32)],
        "coda_set_watchdog_ms": [c_uint32],
        "coda_set_launch_overlap": [c_int32],
        "coda_inject_dropped_stage": [c_int32],
        "coda_device_sm_count": [P(c_int32)],
        "coda_rms_gain": [P(CodaTensor), c_void_p, c_float, c_void_p, P(CodaTensor), c_void_p],
        "coda_xent_combine": [c_void_p, c_void_p, c_int64, c_int32, c_int64, c_void_p, c_void_p, c_int64, c_void_p,
                              c_void_p, c_void_p, c_void_p],
        "coda_lm_head_xent_forward": [P(CodaXentFwd), c_void_p],
        "coda_lm_head_xent_backward": [P(CodaXentBwd), c_void_p],
        "coda_rope_backward": [P(CodaTensor), P(CodaTensor), c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                               c_int64, P(CodaTensor), c_void_p, c_void_p],
        "coda_qkv_rope_backward": [P(CodaQkvRopeBwd), c_void_p],
        "coda_quantize_nvfp4": [P(CodaTensor), c_float, P(CodaTensor), c_void_p, c_void_p, c_void_p],
        "coda_mlp_nvfp4": [P(CodaMlpNvfp4), c_void_p],
        "coda_quantize_nvfp4_t": [P(CodaTensor), c_int32, c_float, P(CodaTensor), c_void_p, P(CodaTensor), c_void_p,
                                  c_void_p, c_void_p],
        "coda_mlp_nvfp4_backward": [P(CodaMlpNvfp4Bwd), c_void_p],
    }
    for name, args in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = c_int32
    L.coda_workspace_size.argtypes = [c_int32, c_int64, c_int64, c_int64]
    L.coda_workspace_size.restype = c_size_t
    L.coda_nvfp4_scale_bytes.argtypes = [c_int64, c_int64]
    L.coda_nvfp4_scale_bytes.restype = c_size_t
    L.coda_status_string.argtypes = [c_int32]
    L.coda_status_string.restype = c_char_p
    L.coda_version.argtypes = []
    L.coda_version.restype = c_char_p
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().coda_status_string(int(status)).decode()


def version() -> str:
    return lib().coda_version().decode()


def _check(status, where):
    if status != OK:
        raise CodaError(int(status), where)


def _stream(stream):
    if stream is None:
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return c_void_p(stream.cuda_stream)
    return c_void_p(int(stream))


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.uint8: E4M3}


def desc(t: torch.Tensor) -> CodaTensor:
    """coda_tensor of a 2-D tensor (layout from its strides)."""
    if t.dim() != 2:
        raise ValueError("coda tensors are 2-D")
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    rows, cols = t.shape
    s0, s1 = t.stride()
    if s1 == 1 or cols <= 1:
        layout, ld = ROW_MAJOR, max(s0, cols, 1)
    elif s0 == 1 or rows <= 1:
        layout, ld = COL_MAJOR, max(s1, rows, 1)
    else:
        raise ValueError("tensor must be row- or column-major (one unit stride)")
    return CodaTensor(c_void_p(t.data_ptr()), _DT[t.dtype], layout, rows, cols, ld)


class Nvfp4:
    """An NVFP4 tensor [R, K]: ``codes`` (uint8 [R, K / 2], two e2m1 codes per byte, element 2j
    in the low nibble of byte j), ``scales`` (uint8, coda_nvfp4_scale_bytes(R, K) bytes in the
    library's block-scale layout) and the fp32 tensor scale ``s``."""

    def __init__(self, codes, scales, s):
        self.codes, self.scales, self.s = codes, scales, float(s)

    @property
    def shape(self):
        return self.codes.shape[0], 2 * self.codes.shape[1]

    @staticmethod
    def empty(R, K, s=1.0, device="cuda"):
        return Nvfp4(torch.empty((R, K // 2), dtype=torch.uint8, device=device),
                     torch.zeros((coda_nvfp4_scale_bytes(R, K),), dtype=torch.uint8, device=device), s)


def desc_nvfp4(codes) -> CodaTensor:
    """coda_tensor of NVFP4 codes held as uint8 [R, K / 2] (row-major)."""
    if codes.dim() != 2 or codes.dtype != torch.uint8 or (codes.shape[0] > 1 and codes.stride(1) != 1):
        raise ValueError("NVFP4 codes are a row-major uint8 [R, K / 2] tensor")
    R, KB = codes.shape
    return CodaTensor(c_void_p(codes.data_ptr()), NVFP4, ROW_MAJOR, R, 2 * KB, 2 * max(codes.stride(0), KB, 1))


def _desc_any(t):
    return desc_nvfp4(t.codes) if isinstance(t, Nvfp4) else desc(t)


def program(*ops) -> CodaProgram:
    if len(ops) > MAX_OPS:
        raise ValueError("too many ops")
    p = CodaProgram()
    p.n_ops = len(ops)
    for i, o in enumerate(ops):
        p.ops[i] = int(o)
    return p


# ------------------------------------------------------------------------ the calls
def coda_gemm_epilogue(A, W, ops, out, *, residual=None, row_scale=None, row_coef=None, col_scale=None,
                       aux_in=None, aux_in2=None, rope_cos=None, rope_sin=None, rope_seq_len=0, rope_head_dim=0,
                       rope_ncols=0, tensor_scale=1.0, out_scale=1.0, row_partials=None, col_partials=None,
                       store_aux=None, amax=None, row_index=None, row_partials2=None, row_values=None,
                       out_shape=None, stream=None):
    """out = epilogue(ops, A . W^T); see include/coda.h for the programs.  For XENT_PARTIAL
    (no output tile) pass out=None and out_shape=(M, V).  A, W (and a SWIGLU out) may be
    Nvfp4 tensors: their block scales ride along, and tensor_scale carries s_A * s_W."""
    keep = []

    def tp(t):
        if t is None:
            return None
        d = desc(t)
        keep.append(d)
        return ctypes.pointer(d)

    sc = lambda t: _ptr(t.scales) if isinstance(t, Nvfp4) else None
    side = CodaSide(tp(residual), _ptr(row_scale), _ptr(row_coef), _ptr(col_scale), tp(aux_in), tp(aux_in2),
                    _ptr(rope_cos), _ptr(rope_sin), rope_seq_len, rope_head_dim, rope_ncols, tensor_scale, out_scale,
                    _ptr(row_index), sc(A), sc(W), out.s if isinstance(out, Nvfp4) else 0.0)
    aux = CodaAux(_ptr(row_partials), row_partials.stride(0) if row_partials is not None else 0,
                  _ptr(col_partials), col_partials.stride(0) if col_partials is not None else 0,
                  tp(store_aux), _ptr(amax), _ptr(row_partials2), _ptr(row_values), sc(out))
    a, w = _desc_any(A), _desc_any(W)
    if out is None:
        o = CodaTensor(None, BF16, ROW_MAJOR, out_shape[0], out_shape[1], max(out_shape[1], 1))
    else:
        o = _desc_any(out)
    prog = program(*ops)
    st = lib().coda_gemm_epilogue(ctypes.byref(a), ctypes.byref(w), ctypes.byref(prog), ctypes.byref(side),
                                  ctypes.byref(o), ctypes.byref(aux), _stream(stream))
    _check(st, "coda_gemm_epilogue")


def coda_rms_partial_reduce(partials, M, d, eps, out, mode=REDUCE_RSQRT_MEAN, rowscale=None, stream=None):
    nparts, ld = partials.shape[0], partials.stride(0)
    st = lib().coda_rms_partial_reduce(_ptr(partials), ld, nparts, M, d, eps, mode, _ptr(rowscale), _ptr(out),
                                       _stream(stream))
    _check(st, "coda_rms_partial_reduce")


def coda_row_rms(X, eps, r_out, stream=None):
    x = desc(X)
    _check(lib().coda_row_rms(ctypes.byref(x), eps, _ptr(r_out), _stream(stream)), "coda_row_rms")


def coda_col_reduce(parts, out, stream=None):
    nblocks, N = parts.shape
    st = lib().coda_col_reduce(_ptr(parts), nblocks, N, parts.stride(0), _ptr(out), _stream(stream))
    _check(st, "coda_col_reduce")


def coda_fold_gain(W, g, W_out, stream=None, out_scale=1.0):
    w, wo = desc(W), desc(W_out)
    st = lib().coda_fold_gain(ctypes.byref(w), _ptr(g), float(out_scale), ctypes.byref(wo), _stream(stream))
    _check(st, "coda_fold_gain")


def coda_rope_table(seq_len, head_dim, base, cos_out, sin_out, stream=None):
    st = lib().coda_rope_table(seq_len, head_dim, base, _ptr(cos_out), _ptr(sin_out), _stream(stream))
    _check(st, "coda_rope_table")


def coda_rms_gain(X, g, eps, r_out, u_out, stream=None):
    x, u = desc(X), desc(u_out)
    _check(lib().coda_rms_gain(ctypes.byref(x), _ptr(g), eps, _ptr(r_out), ctypes.byref(u), _stream(stream)),
           "coda_rms_gain")


def coda_xent_combine(Pm, Ps, target_logit, targets, V, lse, loss, mean=None, stream=None):
    nparts, M = Pm.shape[0], lse.shape[0]
    st = lib().coda_xent_combine(_ptr(Pm), _ptr(Ps), Pm.stride(0), nparts, M, _ptr(target_logit), _ptr(targets), V,
                                 _ptr(lse), _ptr(loss), _ptr(mean), _stream(stream))
    _check(st, "coda_xent_combine")


def coda_lm_head_xent_forward(h, g, W_v, targets, eps, u, r, lse, loss, loss_mean, workspace, stream=None):
    M, H = h.shape
    V = W_v.shape[0]
    io = CodaXentFwd(M, H, V, eps, _ptr(h), _ptr(g), _ptr(W_v), _ptr(targets), _ptr(u), _ptr(r), _ptr(lse),
                     _ptr(loss), _ptr(loss_mean), _ptr(workspace))
    _check(lib().coda_lm_head_xent_forward(ctypes.byref(io), _stream(stream)), "coda_lm_head_xent_forward")


def coda_lm_head_xent_backward(h, g, W_v, targets, u, r, lse, dloss, e, dh, dW_v, dg, c, workspace, stream=None):
    M, H = h.shape
    V = W_v.shape[0]
    io = CodaXentBwd(M, H, V, dloss, _ptr(h), _ptr(g), _ptr(W_v), _ptr(targets), _ptr(u), _ptr(r), _ptr(lse),
                     _ptr(e), _ptr(dh), _ptr(dW_v), _ptr(dg), _ptr(c), _ptr(workspace))
    _check(lib().coda_lm_head_xent_backward(ctypes.byref(io), _stream(stream)), "coda_lm_head_xent_backward")


def coda_rope_backward(dout, out, r, rope_cos, rope_sin, seq_len, head_dim, rope_ncols, H, e_out, c_out,
                       stream=None):
    d, o, e = desc(dout), desc(out), desc(e_out)
    st = lib().coda_rope_backward(ctypes.byref(d), ctypes.byref(o), _ptr(r), _ptr(rope_cos), _ptr(rope_sin), seq_len,
                                  head_dim, rope_ncols, H, ctypes.byref(e), _ptr(c_out), _stream(stream))
    _check(st, "coda_rope_backward")


def coda_qkv_rope_backward(h, g, W_qkv, r, out, dout, seq_len, head_dim, rope_ncols, rope_cos, rope_sin, e, dh,
                           dW_qkv, dg, c, workspace, dres=None, stream=None):
    M, H = h.shape
    N = W_qkv.shape[0]
    io = CodaQkvRopeBwd(M, H, N, seq_len, head_dim, rope_ncols, _ptr(h), _ptr(g), _ptr(W_qkv), _ptr(r), _ptr(out),
                        _ptr(dout), _ptr(dres), _ptr(rope_cos), _ptr(rope_sin), _ptr(e), _ptr(dh), _ptr(dW_qkv),
                        _ptr(dg), _ptr(c), _ptr(workspace))
    _check(lib().coda_qkv_rope_backward(ctypes.byref(io), _stream(stream)), "coda_qkv_rope_backward")


def coda_workspace_size(which, M, H, F):
    return int(lib().coda_workspace_size(which, M, H, F))


def coda_block_forward(O, R, W_o, W_gu, W_d, eps, h, r, a, Y, workspace, Z=None, Y_partials=None, g=None, u=None,
                       stream=None):
    """Block forward.  With g (and the u buffer) the gain is broadcast in G1's epilogue and
    W_gu is the unfolded weight; without g, W_gu must already carry the folded gain."""
    M, H = O.shape
    F = W_d.shape[1]
    io = CodaBlockFwd(M, H, F, eps, _ptr(O), _ptr(R), _ptr(W_o), _ptr(W_gu), _ptr(W_d), _ptr(g), _ptr(u), _ptr(h),
                      _ptr(r), _ptr(a), _ptr(Y), _ptr(Z), _ptr(Y_partials), _ptr(workspace))
    _check(lib().coda_block_forward(ctypes.byref(io), _stream(stream)), "coda_block_forward")


def coda_block_forward_noalloc(O, R, W_o, W_gu, W_d, eps, h, r, a, Y, Z=None, Y_partials=None, g=None, u=None,
                               stream=None):
    """The block forward for callers that cannot allocate device memory: no workspace is
    passed; the chain's partial sums live in the library's static device array (see
    include/coda.h for the size limit and the sharing rules)."""
    M, H = O.shape
    F = W_d.shape[1]
    io = CodaBlockFwd(M, H, F, eps, _ptr(O), _ptr(R), _ptr(W_o), _ptr(W_gu), _ptr(W_d), _ptr(g), _ptr(u), _ptr(h),
                      _ptr(r), _ptr(a), _ptr(Y), _ptr(Z), _ptr(Y_partials), None)
    _check(lib().coda_block_forward_noalloc(ctypes.byref(io), _stream(stream)), "coda_block_forward_noalloc")


def coda_block_backward(O, W_o, W_gu, W_d, g, h, r, Z, a, dY, e, dh, dO, dW_o, dW_gu, dW_d, dg, c, workspace,
                        stream=None):
    M, H = O.shape
    F = W_d.shape[1]
    io = CodaBlockBwd(M, H, F, _ptr(O), _ptr(W_o), _ptr(W_gu), _ptr(W_d), _ptr(g), _ptr(h), _ptr(r), _ptr(Z),
                      _ptr(a), _ptr(dY), _ptr(e), _ptr(dh), _ptr(dO), _ptr(dW_o), _ptr(dW_gu), _ptr(dW_d), _ptr(dg),
                      _ptr(c), _ptr(workspace))
    _check(lib().coda_block_backward(ctypes.byref(io), _stream(stream)), "coda_block_backward")


def coda_qkv_rope(h, W_qkv, eps, seq_len, head_dim, rope_ncols, rope_cos, rope_sin, r, out, stream=None):
    M, H = h.shape
    N = W_qkv.shape[0]
    io = CodaQkvRope(M, H, N, seq_len, head_dim, rope_ncols, eps, _ptr(h), _ptr(W_qkv), _ptr(rope_cos),
                     _ptr(rope_sin), _ptr(r), _ptr(out))
    _check(lib().coda_qkv_rope(ctypes.byref(io), _stream(stream)), "coda_qkv_rope")


def coda_mlp_fp8(h, X_q, W_q, W_dq, s_x, s_w, s_wd, s_a, eps, r, a_q, amax, Y, Y_partials, Z=None, stream=None):
    M, H = h.shape
    F = W_dq.shape[1]
    io = CodaMlpFp8(M, H, F, eps, s_x, s_w, s_wd, s_a, _ptr(h), _ptr(X_q), _ptr(W_q), _ptr(W_dq), _ptr(r),
                    _ptr(a_q), _ptr(amax), _ptr(Y), _ptr(Y_partials), _ptr(Z))
    _check(lib().coda_mlp_fp8(ctypes.byref(io), _stream(stream)), "coda_mlp_fp8")


def coda_mlp_fp8_backward(h, X_q, W_q, W_dq, Z, a_q, r, dY, s_x, s_w, s_wd, s_a, s_dy, s_e, dY_q, amax_dy, e_q,
                          amax_e, c, dh, dW_d, dW, workspace, stream=None):
    M, H = h.shape
    F = W_dq.shape[1]
    io = CodaMlpFp8Bwd(M, H, F, s_x, s_w, s_wd, s_a, s_dy, s_e, _ptr(h), _ptr(X_q), _ptr(W_q), _ptr(W_dq), _ptr(Z),
                       _ptr(a_q), _ptr(r), _ptr(dY), _ptr(dY_q), _ptr(amax_dy), _ptr(e_q), _ptr(amax_e), _ptr(c),
                       _ptr(dh), _ptr(dW_d), _ptr(dW), _ptr(workspace))
    _check(lib().coda_mlp_fp8_backward(ctypes.byref(io), _stream(stream)), "coda_mlp_fp8_backward")


def coda_nvfp4_scale_bytes(R, K):
    return int(lib().coda_nvfp4_scale_bytes(R, K))


def coda_quantize_nvfp4(X, Q, amax=None, stream=None):
    """Q (an Nvfp4 of X's shape, tensor scale Q.s) = NVFP4 quantisation of the bf16 tensor X."""
    x, q = desc(X), desc_nvfp4(Q.codes)
    _check(lib().coda_quantize_nvfp4(ctypes.byref(x), Q.s, ctypes.byref(q), _ptr(Q.scales), _ptr(amax),
                                     _stream(stream)), "coda_quantize_nvfp4")


QT_PLAIN, QT_SWIGLU = 0, 1


def coda_mlp_nvfp4_backward(h, W_guT, W_dT, Z, r, dY, s_x, s_a, s_dy, s_e, dY_r, dY_c, e, e_r, e_c, a_c, x_c, amax_dy,
                            amax_e, c, dh, dW_d, dW, workspace, stream=None):
    """Backward of the NVFP4 MLP.  W_guT, W_dT are the transposed weight quantisations (Nvfp4
    [H, 2F] and [F, H], their .s the tensor scales); dY_r, dY_c, e_r, e_c, a_c, x_c are Nvfp4
    outputs whose .s is ignored (the scales s_dy, s_e, s_a, s_x apply)."""
    M, H = h.shape
    F = Z.shape[1] // 2
    io = CodaMlpNvfp4Bwd(M, H, F, s_x, W_guT.s, W_dT.s, s_a, s_dy, s_e, _ptr(h), _ptr(W_guT.codes),
                         _ptr(W_guT.scales), _ptr(W_dT.codes), _ptr(W_dT.scales), _ptr(Z), _ptr(r), _ptr(dY),
                         _ptr(dY_r.codes), _ptr(dY_r.scales), _ptr(dY_c.codes), _ptr(dY_c.scales), _ptr(e),
                         _ptr(e_r.codes), _ptr(e_r.scales), _ptr(e_c.codes), _ptr(e_c.scales), _ptr(a_c.codes),
                         _ptr(a_c.scales), _ptr(x_c.codes), _ptr(x_c.scales), _ptr(amax_dy), _ptr(amax_e), _ptr(c),
                         _ptr(dh), _ptr(dW_d), _ptr(dW), _ptr(workspace))
    _check(lib().coda_mlp_nvfp4_backward(ctypes.byref(io), _stream(stream)), "coda_mlp_nvfp4_backward")


def coda_quantize_nvfp4_t(X, Q, mode=QT_PLAIN, amax=None, stream=None, Q_rows=None):
    """Q (an Nvfp4 [C, R], tensor scale Q.s) = NVFP4 quantisation of the bf16 X [R, C] along its
    columns, i.e. of X^T; with mode QT_SWIGLU, X is [G | U] ([R, 2C]) and silu(G) U is quantised.
    Q_rows (an Nvfp4 [R, C]) also receives the quantisation along the rows, with the scale Q.s."""
    x, q = desc(X), desc_nvfp4(Q.codes)
    qr = ctypes.byref(desc_nvfp4(Q_rows.codes)) if Q_rows is not None else None
    _check(lib().coda_quantize_nvfp4_t(ctypes.byref(x), int(mode), Q.s, ctypes.byref(q), _ptr(Q.scales), qr,
                                       _ptr(Q_rows.scales) if Q_rows is not None else None, _ptr(amax),
                                       _stream(stream)), "coda_quantize_nvfp4_t")


def coda_mlp_nvfp4(h, X, W, Wd, eps, r, a, amax, Y, Y_partials, stream=None):
    """NVFP4 MLP: X, W (gate/up), Wd and the output a are Nvfp4 tensors;
    a.s is the delayed scale s_a of the SwiGLU output."""
    M, H = h.shape
    F = Wd.shape[1]
    io = CodaMlpNvfp4(M, H, F, eps, X.s, W.s, Wd.s, a.s, _ptr(h), _ptr(X.codes), _ptr(X.scales), _ptr(W.codes),
                      _ptr(W.scales), _ptr(Wd.codes), _ptr(Wd.scales), _ptr(r), _ptr(a.codes), _ptr(a.scales),
                      _ptr(amax), _ptr(Y), _ptr(Y_partials))
    _check(lib().coda_mlp_nvfp4(ctypes.byref(io), _stream(stream)), "coda_mlp_nvfp4")


def coda_quantize_e4m3(X, scale, Q, amax=None, stream=None):
    x, q = desc(X), desc(Q)
    _check(lib().coda_quantize_e4m3(ctypes.byref(x), scale, ctypes.byref(q), _ptr(amax), _stream(stream)),
           "coda_quantize_e4m3")


def coda_get_device_status(stream=None):
    """(status, site): synchronises the stream and reads + clears the device status word."""
    site = c_int32(0)
    st = lib().coda_get_device_status(_stream(stream), ctypes.byref(site))
    return int(st), int(site.value)


def coda_set_launch_overlap(enable):
    _check(lib().coda_set_launch_overlap(1 if enable else 0), "coda_set_launch_overlap")


def coda_set_watchdog_ms(ms):
    _check(lib().coda_set_watchdog_ms(int(ms)), "coda_set_watchdog_ms")


def coda_inject_dropped_stage(enable=True):
    """enable: False / 0 off, True / 1 every producer drops its first k-block, 2 only the
    second CTA of each pair, 3 only the pair's leader."""
    mode = int(enable) if not isinstance(enable, bool) else (1 if enable else 0)
    _check(lib().coda_inject_dropped_stage(mode), "coda_inject_dropped_stage")


def coda_device_sm_count():
    n = c_int32(0)
    _check(lib().coda_device_sm_count(ctypes.byref(n)), "coda_device_sm_count")
    return int(n.value)
