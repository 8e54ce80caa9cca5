"""The C ABI without a GPU: the library loads, exports every function include/coda.h
declares, and rejects bad arguments on the host before touching a device.  No compute call
runs here; a well-formed call on a machine without an sm_103 device returns
CODA_ERR_NO_DEVICE (there is no CPU fallback)."""
import ctypes
import os
import re

import pytest

from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "coda.h")) as f:
        txt = f.read()
    return sorted(set(re.findall(r"CODA_API\s+[\w\s\*]+?\b(coda_\w+)\s*\(", txt)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(C.LIB_PATH):
        from gemm_epilogue_transformer_tcgen05_gb300 import build
        build.build()
    return C.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 17
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(C.EXPORTED)


def test_status_strings_and_version(L):
    assert C.version().startswith("coda-gb300")
    for s in range(-8, 1):
        assert C.status_string(s) != "unknown status"
    assert C.status_string(-99) == "unknown status"


def test_workspace_sizes(L):
    assert C.coda_workspace_size(C.WS_BLOCK_FWD, 16384, 2048, 8192) == 8 * 16384 * 4
    assert C.coda_workspace_size(C.WS_BLOCK_BWD, 16384, 2048, 8192) == (32 * 16384 + 512 * 2048) * 4
    assert C.coda_workspace_size(C.WS_BLOCK_BWD, 300, 256, 384) == (2 * 300 + 10 * 256) * 4
    assert C.coda_workspace_size(7, 1, 1, 1) == 0


def _t(ptr, dtype, rows, cols, ld, layout=C.ROW_MAJOR):
    return C.CodaTensor(ctypes.c_void_p(ptr), dtype, layout, rows, cols, ld)


def _call(A, W, ops, out, side=None, aux=None):
    p = C.program(*ops)
    return C.lib().coda_gemm_epilogue(ctypes.byref(A) if A else None, ctypes.byref(W) if W else None,
                                      ctypes.byref(p), ctypes.byref(side) if side else None,
                                      ctypes.byref(out) if out else None, ctypes.byref(aux) if aux else None, None)


FAKE = 0x10000   # never dereferenced: every check below fails before any device access


def test_host_validation_codes(L):
    A = _t(FAKE, C.BF16, 256, 512, 512)
    W = _t(FAKE, C.BF16, 256, 512, 512)
    out = _t(FAKE, C.BF16, 256, 256, 256)
    assert _call(None, W, [], out) == C.ERR_NULL
    assert _call(A, W, [C.OP_ROW_SUMSQ_PARTIAL, C.OP_ADD_SIDE], out) == C.ERR_UNSUPPORTED_PROGRAM
    assert _call(A, W, [C.OP_SWIGLU, C.OP_ROW_SCALE], out) == C.ERR_UNSUPPORTED_PROGRAM
    assert _call(A, _t(FAKE, C.BF16, 256, 256, 512), [], out) == C.ERR_SHAPE         # K mismatch
    assert _call(A, W, [], _t(FAKE, C.BF16, 256, 128, 256)) == C.ERR_SHAPE          # N mismatch
    assert _call(_t(FAKE + 8, C.BF16, 256, 512, 512), W, [], out) == C.ERR_ALIGN    # base
    assert _call(_t(FAKE, C.BF16, 256, 500, 500), _t(FAKE, C.BF16, 256, 500, 500), [], out) == C.ERR_ALIGN
    assert _call(A, _t(FAKE, C.F32, 256, 512, 512), [], out) == C.ERR_DTYPE          # mixed operands
    assert _call(A, W, [C.OP_ROW_SCALE], out) == C.ERR_NULL                          # r missing
    assert _call(A, W, [C.OP_ADD_SIDE], out) == C.ERR_NULL                           # residual missing
    swo = _t(FAKE, C.BF16, 256, 200, 200)                                            # SWIGLU N % 128
    assert _call(A, _t(FAKE, C.BF16, 400, 512, 512), [C.OP_SWIGLU], swo) == C.ERR_SHAPE
    empty = _t(0, C.BF16, 0, 512, 512)
    assert _call(empty, W, [], _t(0, C.BF16, 0, 256, 256)) == C.OK                   # M = 0: no-op


def test_well_formed_call_without_device_is_refused(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    A = _t(FAKE, C.BF16, 256, 512, 512)
    W = _t(FAKE, C.BF16, 256, 512, 512)
    out = _t(FAKE, C.BF16, 256, 256, 256)
    assert _call(A, W, [], out) == C.ERR_NO_DEVICE
    n = ctypes.c_int32(0)
    assert L.coda_device_sm_count(ctypes.byref(n)) == C.ERR_NO_DEVICE


def test_other_entry_points_validate(L):
    assert L.coda_rms_partial_reduce(None, 1, 1, 1, 1, 1e-6, 0, None, None, None) == C.ERR_NULL
    assert L.coda_rms_partial_reduce(ctypes.c_void_p(FAKE), 4, 1, 8, 1, 1e-6, 0, None, ctypes.c_void_p(FAKE),
                                     None) == C.ERR_SHAPE                              # ld < M
    assert L.coda_rms_partial_reduce(ctypes.c_void_p(FAKE), 8, 1, 8, 1, 1e-6, 1, None, ctypes.c_void_p(FAKE),
                                     None) == C.ERR_NULL                               # SCALE_SUM needs r
    assert L.coda_col_reduce(None, 1, 1, 1, None, None) == C.ERR_NULL
    assert L.coda_rope_table(0, 64, 1e4, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), None) == C.ERR_SHAPE
    W = _t(FAKE, C.BF16, 16, 12, 12)
    assert L.coda_fold_gain(ctypes.byref(W), ctypes.c_void_p(FAKE), 1.0, ctypes.byref(W), None) == C.ERR_ALIGN
    Wb = _t(FAKE, C.BF16, 16, 32, 32)
    g = ctypes.c_void_p(FAKE + 0x4000)
    fold = lambda w, s, wo: L.coda_fold_gain(ctypes.byref(w), g, s, ctypes.byref(wo), None)
    assert fold(Wb, 0.0, Wb) == C.ERR_SHAPE                                        # out_scale must be > 0
    assert fold(Wb, float("inf"), Wb) == C.ERR_SHAPE
    assert fold(Wb, 1.0, _t(FAKE + 0x8000, C.F32, 16, 32, 32)) == C.ERR_DTYPE       # bf16 -> fp32
    assert fold(Wb, 1.0, _t(FAKE, C.E4M3, 16, 32, 32)) == C.ERR_SHAPE              # e4m3 out in place
    assert fold(_t(FAKE, C.BF16, 16, 24, 32), 1.0, _t(FAKE + 0x8000, C.E4M3, 16, 24, 32)) == C.ERR_SHAPE  # K % 16
    assert fold(Wb, 1.0, _t(FAKE + 0x8000, C.E4M3, 16, 16, 32)) == C.ERR_SHAPE    # shapes differ
    assert L.coda_fold_gain(None, g, 1.0, ctypes.byref(Wb), None) == C.ERR_NULL
    assert L.coda_block_forward(None, None) == C.ERR_NULL
    assert L.coda_block_backward(None, None) == C.ERR_NULL
    assert L.coda_qkv_rope(None, None) == C.ERR_NULL
    assert L.coda_mlp_fp8(None, None) == C.ERR_NULL
    assert L.coda_set_watchdog_ms(0) == C.ERR_SHAPE
    assert L.coda_get_device_status(None, None) == C.ERR_NULL


def test_fp8_backward_quantiser_and_overlap_validate(L):
    X = _t(FAKE, C.BF16, 64, 48, 48)
    Q = _t(FAKE, C.E4M3, 64, 48, 48)
    assert L.coda_quantize_e4m3(None, 1.0, ctypes.byref(Q), None, None) == C.ERR_NULL
    assert L.coda_quantize_e4m3(ctypes.byref(X), 0.0, ctypes.byref(Q), None, None) == C.ERR_SHAPE   # scale > 0
    assert L.coda_quantize_e4m3(ctypes.byref(Q), 1.0, ctypes.byref(Q), None, None) == C.ERR_DTYPE   # bf16 in
    assert L.coda_quantize_e4m3(ctypes.byref(X), 1.0, ctypes.byref(_t(FAKE, C.E4M3, 64, 32, 48)), None,
                                None) == C.ERR_SHAPE
    assert L.coda_quantize_e4m3(ctypes.byref(_t(FAKE, C.BF16, 64, 40, 40)), 1.0,
                                ctypes.byref(_t(FAKE, C.E4M3, 64, 40, 48)), None, None) == C.ERR_SHAPE   # N % 16
    assert L.coda_mlp_fp8_backward(None, None) == C.ERR_NULL
    f = ctypes.c_void_p(FAKE)
    io = C.CodaMlpFp8Bwd(M=256, H=256, F=128, s_x=1.0, s_w=1.0, s_wd=1.0, s_a=1.0, s_dy=1.0, s_e=0.0, h=f, X_q=f,
                         W_q=f, W_dq=f, Z=f, a_q=f, r=f, dY=f, dY_q=f, amax_dy=f, e_q=f, amax_e=f, c=f, dh=f,
                         dW_d=f, dW=f, workspace=f)
    assert L.coda_mlp_fp8_backward(ctypes.byref(io), None) == C.ERR_SHAPE            # s_e must be > 0
    io.s_e, io.F = 1.0, 100
    assert L.coda_mlp_fp8_backward(ctypes.byref(io), None) == C.ERR_SHAPE            # F % 128
    io.F, io.dW = 128, None
    assert L.coda_mlp_fp8_backward(ctypes.byref(io), None) == C.ERR_NULL
    assert C.coda_workspace_size(C.WS_MLP_FP8_BWD, 16384, 4096, 14336) == 56 * 16384 * 4
    assert L.coda_set_launch_overlap(2) == C.ERR_SHAPE
    assert L.coda_set_launch_overlap(1) == C.OK


def test_binding_reads_layout_from_strides():
    import torch
    x = torch.empty((64, 32), dtype=torch.bfloat16)
    d = C.desc(x)
    assert (d.layout, d.rows, d.cols, d.ld) == (C.ROW_MAJOR, 64, 32, 32)
    d = C.desc(x.t())
    assert (d.layout, d.rows, d.cols, d.ld) == (C.COL_MAJOR, 32, 64, 32)
    with pytest.raises(ValueError):
        C.desc(torch.empty((4, 4, 4)))


def test_nvfp4_entry_points_validate(L):
    f = ctypes.c_void_p(FAKE)
    assert C.coda_nvfp4_scale_bytes(300, 512) == 3 * 8 * 512
    assert C.coda_nvfp4_scale_bytes(0, 512) == 0
    X = _t(FAKE, C.BF16, 256, 512, 512)
    Q = _t(FAKE, C.NVFP4, 256, 512, 512)
    q = L.coda_quantize_nvfp4
    assert q(None, 1.0, ctypes.byref(Q), f, None, None) == C.ERR_NULL
    assert q(ctypes.byref(X), 1.0, ctypes.byref(Q), None, None, None) == C.ERR_NULL        # scales missing
    assert q(ctypes.byref(X), 0.0, ctypes.byref(Q), f, None, None) == C.ERR_SHAPE         # s > 0
    assert q(ctypes.byref(X), 1.0, ctypes.byref(X), f, None, None) == C.ERR_DTYPE         # Q must be NVFP4
    assert q(ctypes.byref(X), 1.0, ctypes.byref(Q), ctypes.c_void_p(FAKE + 8), None, None) == C.ERR_ALIGN
    assert q(ctypes.byref(_t(FAKE, C.BF16, 256, 48, 48)), 1.0, ctypes.byref(_t(FAKE, C.NVFP4, 256, 48, 64)), f,
             None, None) == C.ERR_SHAPE                                                     # K % 64
    assert q(ctypes.byref(X), 1.0, ctypes.byref(_t(FAKE, C.NVFP4, 256, 512, 520)), f, None,
             None) == C.ERR_ALIGN                                                           # ld / 2 % 16
    # the GEMM with NVFP4 operands
    A = _t(FAKE, C.NVFP4, 256, 512, 512)
    W = _t(FAKE, C.NVFP4, 256, 512, 512)
    out = _t(FAKE, C.F32, 256, 256, 256)
    p = C.program(C.OP_TENSOR_SCALE)
    side = C.CodaSide()
    aux = C.CodaAux()
    g = lambda A_, W_, o: L.coda_gemm_epilogue(ctypes.byref(A_), ctypes.byref(W_), ctypes.byref(p), ctypes.byref(side),
                                               ctypes.byref(o), ctypes.byref(aux), None)
    assert g(A, W, out) == C.ERR_NULL                                                         # block scales missing
    side.a_block_scales, side.w_block_scales = FAKE, FAKE + 8
    assert g(A, W, out) == C.ERR_ALIGN
    side.w_block_scales = FAKE
    assert g(_t(FAKE, C.NVFP4, 256, 320, 320), _t(FAKE, C.NVFP4, 256, 320, 320), out) == C.ERR_SHAPE   # K % 256
    assert g(A, _t(FAKE, C.BF16, 256, 512, 512), out) == C.ERR_DTYPE                          # mixed operands
    assert g(A, W, _t(FAKE, C.NVFP4, 256, 256, 256)) == C.ERR_DTYPE                           # fp4 out: SWIGLU only
    assert g(_t(FAKE, C.NVFP4, 256, 512, 512, C.COL_MAJOR), W, out) == C.ERR_SHAPE            # row-major only
    # the chain
    assert L.coda_mlp_nvfp4(None, None) == C.ERR_NULL
    io = C.CodaMlpNvfp4(M=256, H=512, F=512, eps=1e-6, s_x=1.0, s_w=1.0, s_wd=1.0, s_a=1.0, h=f, X_q=f, X_sf=f,
                        W_q=f, W_sf=f, W_dq=f, W_dsf=f, r=f, a_q=f, a_sf=f, amax=f, Y=f, Y_partials=f)
    io.F = 384
    assert L.coda_mlp_nvfp4(ctypes.byref(io), None) == C.ERR_SHAPE                            # F % 256
    io.F, io.s_a = 512, 0.0
    assert L.coda_mlp_nvfp4(ctypes.byref(io), None) == C.ERR_SHAPE                            # s_a > 0
    io.s_a, io.W_dsf = 1.0, None
    assert L.coda_mlp_nvfp4(ctypes.byref(io), None) == C.ERR_NULL
    io.W_dsf, io.M = f, 0
    assert L.coda_mlp_nvfp4(ctypes.byref(io), None) == C.OK                                   # empty batch: no-op


def test_nvfp4_backward_entry_points_validate(L):
    f = ctypes.c_void_p(FAKE)
    qt = L.coda_quantize_nvfp4_t
    X = _t(FAKE, C.BF16, 256, 384, 384)
    Qc = _t(FAKE, C.NVFP4, 384, 256, 256)          # X^T
    Qr = _t(FAKE, C.NVFP4, 256, 384, 384)
    assert qt(None, 0, 1.0, ctypes.byref(Qc), f, None, None, None, None) == C.ERR_NULL
    assert qt(ctypes.byref(X), 0, 1.0, ctypes.byref(Qc), None, None, None, None, None) == C.ERR_NULL  # scales missing
    assert qt(ctypes.byref(X), 2, 1.0, ctypes.byref(Qc), f, None, None, None, None) == C.ERR_SHAPE    # mode
    assert qt(ctypes.byref(X), 0, 0.0, ctypes.byref(Qc), f, None, None, None, None) == C.ERR_SHAPE    # s > 0
    assert qt(ctypes.byref(X), 0, 1.0, ctypes.byref(Qr), f, None, None, None, None) == C.ERR_SHAPE    # not X^T
    assert qt(ctypes.byref(X), 1, 1.0, ctypes.byref(Qc), f, None, None, None, None) == C.ERR_SHAPE    # SwiGLU: C = 192
    assert qt(ctypes.byref(X), 0, 1.0, ctypes.byref(Qc), ctypes.c_void_p(FAKE + 8), None, None, None,
              None) == C.ERR_ALIGN
    assert qt(ctypes.byref(X), 0, 1.0, ctypes.byref(Qc), f, ctypes.byref(Qc), f, None, None) == C.ERR_SHAPE  # rows: [R, C]
    assert qt(ctypes.byref(X), 0, 1.0, ctypes.byref(Qc), f, ctypes.byref(Qr), None, None, None) == C.ERR_NULL
    X2 = _t(FAKE, C.BF16, 320, 384, 384)           # R % 128 != 0: no row output
    assert qt(ctypes.byref(X2), 0, 1.0, ctypes.byref(_t(FAKE, C.NVFP4, 384, 320, 320)), f,
              ctypes.byref(_t(FAKE, C.NVFP4, 320, 384, 384)), f, None, None) == C.ERR_SHAPE
    assert qt(ctypes.byref(_t(FAKE, C.BF16, 200, 384, 384)), 0, 1.0, ctypes.byref(_t(FAKE, C.NVFP4, 384, 200, 256)),
              f, None, None, None, None) == C.ERR_SHAPE                                   # R % 64
    # the chain
    assert L.coda_mlp_nvfp4_backward(None, None) == C.ERR_NULL
    names = [n for n, _ in C.CodaMlpNvfp4Bwd._fields_[9:]]
    io = C.CodaMlpNvfp4Bwd(256, 512, 512, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, *([f] * len(names)))
    io.M = 320
    assert L.coda_mlp_nvfp4_backward(ctypes.byref(io), None) == C.ERR_SHAPE        # M % 256
    io.M, io.F = 256, 384
    assert L.coda_mlp_nvfp4_backward(ctypes.byref(io), None) == C.ERR_SHAPE        # F % 256
    io.F, io.s_e = 512, 0.0
    assert L.coda_mlp_nvfp4_backward(ctypes.byref(io), None) == C.ERR_SHAPE        # scales > 0
    io.s_e, io.e_c = 1.0, None
    assert L.coda_mlp_nvfp4_backward(ctypes.byref(io), None) == C.ERR_NULL
    io.e_c, io.workspace = f, ctypes.c_void_p(FAKE + 4)
    assert L.coda_mlp_nvfp4_backward(ctypes.byref(io), None) == C.ERR_ALIGN
    assert C.coda_workspace_size(C.WS_MLP_NVFP4_BWD, 16384, 4096, 14336) == (14336 // 128) * 16384 * 4
