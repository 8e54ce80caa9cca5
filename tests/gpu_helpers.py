"""Shared helpers of the GPU parity tests: device tensors, oracle-side float64 copies and
the tolerance of the parity bar (max relative error with an RMS floor, 2e-2 for bf16 and
tf32 outputs, 6e-2 for the fp8 path)."""
import numpy as np
import torch

import oracle as O

TOL_BF16 = 2e-2
TOL_FP8 = 6e-2


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a tensor (bf16/fp32/e4m3 values are all representable)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def dev(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda").contiguous()


def seeded(shape, seed, std=1.0, mean=0.0, dtype=torch.float32):
    gen = torch.Generator().manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32).normal_(0.0, 1.0, generator=gen) * std + mean
    return t.to(dtype)


def assert_close(got, ref, tol, what):
    err = O.max_rel_err(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"
    return err


def fresh_status():
    """Reads and clears the device status word; asserts no kernel wait ran out of time."""
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
    st, site = C.coda_get_device_status()
    assert st == C.OK, f"device status {st} (site {site})"


def assert_e4m3_codes(codes: np.ndarray, x_ref: np.ndarray, what: str, rel=1e-3):
    """An e4m3 code is a rounding decision the GPU takes in fp32: each code must be one of
    the e4m3 neighbours of the oracle's value x within a relative accumulation error `rel`
    (so only values within that distance of a rounding midpoint may round the other way),
    and almost all codes must equal the oracle's own rounding."""
    v = O.e4m3_decode(codes)
    slack = rel * np.abs(x_ref) + 1e-9
    lo, hi = O.e4m3_round(x_ref - slack), O.e4m3_round(x_ref + slack)
    bad = ~((v >= lo) & (v <= hi))
    assert not bad.any(), f"{what}: {int(bad.sum())} codes outside the rounding window"
    exact = np.mean(v == O.e4m3_round(x_ref))
    assert exact >= 0.999, f"{what}: only {exact:.5f} of the codes equal the oracle's rounding"


def assert_product_close(got, ref, sim, what, factor=1.5):
    """Chain tensors built from products of two bf16-rounded GEMM results (a, e and the
    weight gradients formed from them): max |err| / max |ref| <= 2e-2, and the element-wise
    error (RMS floor) at most `factor` times that of the bf16-storage model (tests/storage_sim)
    on the same elements, and never required below the 2e-2 bar."""
    from tests.storage_sim import normwise
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    nw = normwise(got, ref)
    assert nw <= TOL_BF16, f"{what}: normwise err {nw:.3e} > {TOL_BF16:.1e}"
    el, el_sim = O.max_rel_err(got, ref), O.max_rel_err(sim, ref)
    bound = max(TOL_BF16, factor * el_sim)
    assert el <= bound, f"{what}: element-wise err {el:.3e} > {bound:.3e} (bf16-storage model {el_sim:.3e})"
    return el, el_sim


def nvfp4_window(got_q, got_sf, x, s, rel):
    """NVFP4 codes and block scales are rounding decisions the GPU takes in fp32; the oracle
    takes them in float64 on the plain definition.  Each block scale must lie between the e4m3
    roundings of amax / (6 s) moved by `rel` either way, and each code between the e2m1
    roundings of x / (sf s) moved by `rel` either way, sf being the GPU's own block scale (so a
    block whose scale rounded the other way is still checked, against that scale).  Where that
    window holds a single value (the value is not within `rel` of a rounding midpoint) the
    GPU's decision must therefore equal the oracle's; only the ambiguous ones may differ.
    Returns the fractions of block scales and of codes equal to the oracle's rounding, the
    fraction of codes whose window is ambiguous, and the same for the block scales."""
    R, K = x.shape
    q, sf = O.nvfp4_quantize(x, s)
    amax_b = np.max(np.abs(x).reshape(R, K // 16, 16), axis=2)
    u = amax_b / (6.0 * s)
    lo, hi = O.e4m3_round(u * (1 - rel)), O.e4m3_round(u * (1 + rel))
    bad_sf = ~((got_sf >= lo) & (got_sf <= hi))
    assert not bad_sf.any(), f"{int(bad_sf.sum())} block scales outside the rounding window"
    d = s * np.repeat(got_sf, 16, axis=1)
    y = np.where(d > 0, x / np.where(d > 0, d, 1.0), 0.0)
    slack = rel * np.abs(y)
    qlo, qhi = O.e2m1_round(y - slack), O.e2m1_round(y + slack)
    bad_q = ~((got_q >= qlo) & (got_q <= qhi))
    assert not bad_q.any(), f"{int(bad_q.sum())} codes outside the rounding window"
    same_scale = np.repeat(got_sf == sf, 16, axis=1)
    clear = (qlo == qhi) & same_scale
    assert np.all((got_q == q)[clear]), "a code away from every rounding midpoint differs from the oracle's"
    return (float(np.mean(got_sf == sf)), float(np.mean(got_q == q)), float(np.mean(qlo != qhi)),
            float(np.mean(lo != hi)))
