"""Plants plausible mistakes in the oracle (on the CPU, by monkeypatching a copy of one of
its functions) and checks that at least one pin fails for each.  This shows the pins are
sharp enough to catch a dropped term, a wrong sign or index, or a transposed operand."""
import numpy as np
import pytest

import oracle as O
import oracle.coda_oracle as OC
import tests.test_oracle_pins as pins


def _plant(monkeypatch, name, fn):
    # the pins use the package namespace; internal calls use the module's
    monkeypatch.setattr(O, name, fn)
    monkeypatch.setattr(OC, name, fn)


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_dropped_eps_is_caught(monkeypatch):
    def no_eps(h, eps):
        with np.errstate(divide="ignore"):   # a zero row divides by zero: that is the planted mistake
            return 1.0 / np.sqrt(np.mean(np.asarray(h, float) ** 2, axis=1))
    _plant(monkeypatch, "rms_scale", no_eps)
    assert _fails(pins.test_rms_eps_only_row) or _fails(pins.test_rms_constant_row)


def test_transposed_weight_is_caught(monkeypatch):
    _plant(monkeypatch, "linear", lambda X, W: np.asarray(X, float) @ np.asarray(W, float))
    assert _fails(pins.test_linear_uses_out_in_layout)


def test_wrong_rope_sign_is_caught(monkeypatch):
    orig = O.rope_rotate

    def bad(Z, positions, n_rot_cols, head_dim, base):
        return orig(Z, -np.asarray(positions, float), n_rot_cols, head_dim, base)

    _plant(monkeypatch, "rope_rotate", bad)
    assert _fails(pins.test_rope_closed_form_first_pair)


def test_rope_wrong_pairing_is_caught(monkeypatch):
    def half_split(Z, positions, n_rot_cols, head_dim, base):   # (p, p + hd/2) pairing
        Z = np.asarray(Z, float)
        out = Z.copy()
        phi = np.asarray(positions, float)[:, None] * O.rope_inv_freq(head_dim, base)[None, :]
        c, s = np.cos(phi), np.sin(phi)
        for h0 in range(0, n_rot_cols, head_dim):
            x0 = Z[:, h0:h0 + head_dim // 2]
            x1 = Z[:, h0 + head_dim // 2:h0 + head_dim]
            out[:, h0:h0 + head_dim // 2] = x0 * c - x1 * s
            out[:, h0 + head_dim // 2:h0 + head_dim] = x0 * s + x1 * c
        return out

    _plant(monkeypatch, "rope_rotate", half_split)
    assert _fails(pins.test_rope_closed_form_first_pair)


def test_dropped_residual_grad_is_caught(monkeypatch):
    orig = O.block_backward

    def bad(fwd, Oa, W_o, g, W_gu, W_d, dY):
        out = orig(fwd, Oa, W_o, g, W_gu, W_d, dY)
        dh = out["dh"] - np.asarray(dY, float)
        out.update(dh=dh, dR=dh, dO=dh @ np.asarray(W_o, float), dW_o=dh.T @ np.asarray(Oa, float))
        return out

    _plant(monkeypatch, "block_backward", bad)
    assert _fails(pins.test_backward_matches_finite_differences)


def test_sigmoid_sign_flip_is_caught(monkeypatch):
    _plant(monkeypatch, "sigmoid", lambda x: 1.0 / (1.0 + np.exp(np.asarray(x, float))))
    assert _fails(pins.test_sigmoid_closed_forms_and_symmetry)
    assert _fails(pins.test_silu_closed_forms)


def test_swapped_gate_up_is_caught(monkeypatch):
    _plant(monkeypatch, "swiglu", lambda G, U: O.silu(U) * np.asarray(G, float))
    assert _fails(pins.test_swiglu_gate_and_up_roles)


def test_e4m3_ties_away_is_caught(monkeypatch):
    def away(x):
        x = np.asarray(x, float)
        a = np.minimum(np.abs(x), 448.0)
        _, ex = np.frexp(a)
        q = np.exp2(np.maximum(ex - 1.0, -6.0) - 3.0)
        return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), x)

    _plant(monkeypatch, "e4m3_round", away)
    assert _fails(pins.test_e4m3_ties_to_even_and_saturation)


def test_partial_tile_off_by_one_is_caught(monkeypatch):
    def bad(h, bn):
        h = np.asarray(h, float)
        n = (h.shape[1] + bn - 1) // bn
        return np.stack([np.sum(h[:, t * bn:(t + 1) * bn - 1] ** 2, axis=1) for t in range(n)])

    _plant(monkeypatch, "partial_sumsq", bad)
    assert _fails(pins.test_partials_sum_to_row_sumsq, 64)


def test_xent_target_off_by_one_is_caught(monkeypatch):
    orig = O.cross_entropy

    def bad(logits, targets):
        return orig(logits, (np.asarray(targets) + 1) % np.asarray(logits).shape[1])

    _plant(monkeypatch, "cross_entropy", bad)
    assert _fails(pins.test_cross_entropy_closed_forms)


def test_xent_missing_mean_scale_is_caught(monkeypatch):
    orig = O.lm_head_xent_backward

    def bad(fwd, h, g, W_v, targets, dloss=1.0):
        out = orig(fwd, h, g, W_v, targets, dloss)
        M = np.asarray(h).shape[0]
        return {k: v * M for k, v in out.items()}

    _plant(monkeypatch, "lm_head_xent_backward", bad)
    assert _fails(pins.test_lm_head_xent_backward_matches_finite_differences)


def test_xent_combine_without_rescale_is_caught(monkeypatch):
    _plant(monkeypatch, "xent_combine", lambda m, s: np.max(m, axis=0) + np.log(np.sum(s, axis=0)))
    assert _fails(pins.test_xent_partials_combine_to_logsumexp)


def test_rope_backward_with_forward_rotation_is_caught(monkeypatch):
    orig = O.qkv_rope_backward

    def bad(h, g, W_qkv, dout, eps, seq_len, n_rot_cols, head_dim, base):
        # rotate the gradient by +phi instead of -phi: the transpose of the rotation is missed
        M = np.asarray(h).shape[0]
        pos = np.arange(M) % seq_len
        d2 = O.rope_rotate(O.rope_rotate(dout, pos, n_rot_cols, head_dim, base), pos, n_rot_cols, head_dim, base)
        return orig(h, g, W_qkv, d2, eps, seq_len, n_rot_cols, head_dim, base)

    _plant(monkeypatch, "qkv_rope_backward", bad)
    assert _fails(pins.test_qkv_rope_backward_matches_finite_differences)


def _plant_fp8_bwd(monkeypatch, edit):
    orig = O.mlp_fp8_backward

    def bad(*a, **k):
        return edit(orig(*a, **k), *a, **k)

    _plant(monkeypatch, "mlp_fp8_backward", bad)


def test_fp8_backward_dropped_norm_term_is_caught(monkeypatch):
    def edit(out, *a, **k):
        out["dh"] = out["dh"] + out["c"][:, None] * np.asarray(k.get("h", a[0] if a else None), float)
        return out

    _plant_fp8_bwd(monkeypatch, edit)
    assert _fails(pins.test_mlp_fp8_backward_identity_quantiser_matches_finite_differences)


def test_fp8_backward_missing_e_scale_is_caught(monkeypatch):
    def edit(out, *a, **k):
        s_e = k["s_e"] if "s_e" in k else a[13]
        out["t"] = out["t"] / s_e
        out["dW"] = out["dW"] / s_e
        return out

    _plant_fp8_bwd(monkeypatch, edit)
    assert _fails(pins.test_mlp_fp8_backward_power_of_two_rescaling_is_exact)


def test_fp8_backward_weight_gradient_from_h_is_caught(monkeypatch):
    def edit(out, *a, **k):
        h = np.asarray(k["h"] if "h" in k else a[0], float)
        out["dW"] = out["e_hat"].T @ h
        return out

    _plant_fp8_bwd(monkeypatch, edit)
    assert _fails(pins.test_mlp_fp8_backward_zero_operands_give_closed_forms)


def test_fp8_backward_unquantised_e_is_caught(monkeypatch):
    def edit(out, *a, **k):
        s_e = k["s_e"] if "s_e" in k else a[13]
        out["eq_val"] = out["e"] / s_e
        return out

    _plant_fp8_bwd(monkeypatch, edit)
    assert _fails(pins.test_mlp_fp8_backward_quantises_like_the_library_cast)


# ------------------------------------------------------------------ NVFP4 (reading 9)
import tests.test_oracle_nvfp4 as fp4pins


def test_e2m1_ties_away_is_caught(monkeypatch):
    def away(x):
        x = np.asarray(x, float)
        a = np.minimum(np.abs(x), 6.0)
        _, ex = np.frexp(a)
        q = np.exp2(np.maximum(ex - 1.0, 0.0) - 1.0)
        return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 6.0), x)

    _plant(monkeypatch, "e2m1_round", away)
    assert _fails(fp4pins.test_e2m1_round_is_the_nearest_value_with_ties_to_even)


def test_nvfp4_block_of_32_is_caught(monkeypatch):
    monkeypatch.setattr(OC, "NVFP4_BLOCK", 32)
    assert _fails(fp4pins.test_nvfp4_blocks_are_16_consecutive_elements_of_a_row)


def test_nvfp4_scale_from_e4m3_range_is_caught(monkeypatch):
    # block scale amax / 448 (the e4m3 range) instead of amax / 6 (the e2m1 range)
    def bad(x, s):
        x = np.asarray(x, dtype=float)
        R, K = x.shape
        xb = x.reshape(R, K // 16, 16)
        sf = O.e4m3_round(np.max(np.abs(xb), axis=2) / (448.0 * s))
        d = (sf * s)[:, :, None]
        y = np.where(d > 0, xb / np.where(d > 0, d, 1), 0)
        return O.e2m1_round(y).reshape(R, K), sf

    _plant(monkeypatch, "nvfp4_quantize", bad)
    assert _fails(fp4pins.test_nvfp4_exactly_representable_blocks_round_trip)


def test_nvfp4_scales_repeated_across_rows_is_caught(monkeypatch):
    # block scales spread along the wrong axis (a transposed scale matrix)
    def bad(q, sf, s):
        q, sf = np.asarray(q, float), np.asarray(sf, float)
        R, K = q.shape
        flat = np.repeat(sf.T.ravel(), 16)[: R * K].reshape(R, K)
        return float(s) * flat * q

    _plant(monkeypatch, "nvfp4_dequantize", bad)
    assert _fails(fp4pins.test_block_scaled_gemm_is_the_sum_of_per_block_products)


def test_fold_gain_divided_is_caught(monkeypatch):
    _plant(monkeypatch, "fold_gain", lambda W, g: np.asarray(W, float) / np.asarray(g, float)[None, :])
    assert _fails(pins.test_fold_gain_equals_scaling_input)


def test_silu_grad_missing_term_is_caught(monkeypatch):
    _plant(monkeypatch, "silu_grad", lambda x: O.sigmoid(x))   # drops the x sigma (1 - sigma) term
    assert _fails(pins.test_silu_grad_finite_difference)


def test_logsumexp_without_the_max_shift_is_caught(monkeypatch):
    def unshifted(z):
        with np.errstate(over="ignore"):   # exp(1000) overflows: that is the planted mistake
            return np.log(np.sum(np.exp(np.asarray(z, float)), axis=1))
    _plant(monkeypatch, "logsumexp", unshifted)
    assert _fails(pins.test_logsumexp_matches_scipy_and_closed_forms)


def test_rms_from_partials_over_the_tile_count_is_caught(monkeypatch):
    # mean over the number of partials instead of over d
    _plant(monkeypatch, "rms_scale_from_partials",
           lambda P, d, eps: 1.0 / np.sqrt(np.sum(np.asarray(P, float), axis=0) / np.asarray(P).shape[0] + eps))
    assert _fails(pins.test_partials_sum_to_row_sumsq, 256)


def test_xent_partials_dropping_the_ragged_tile_is_caught(monkeypatch):
    def full_tiles_only(z, bn):
        z = np.asarray(z, float)
        n = z.shape[1] // bn                # the last, partial tile is lost
        blocks = [z[:, t * bn:(t + 1) * bn] for t in range(n)]
        m = np.stack([b.max(axis=1) for b in blocks])
        s = np.stack([np.exp(b - mb[:, None]).sum(axis=1) for b, mb in zip(blocks, m)])
        return m, s
    _plant(monkeypatch, "xent_partials", full_tiles_only)
    assert _fails(pins.test_xent_partials_combine_to_logsumexp)


def test_rope_frequency_without_the_factor_two_is_caught(monkeypatch):
    # theta_p = base^(-p / head_dim) instead of base^(-2p / head_dim)
    _plant(monkeypatch, "rope_inv_freq", lambda head_dim, base: float(base) ** (-np.arange(head_dim // 2) / head_dim))
    assert _fails(pins.test_rope_closed_form_first_pair)


@pytest.mark.parametrize("dropped", ["s_x", "s_wd", "s_a"])
def test_mlp_fp8_dropped_tensor_scale_is_caught(monkeypatch, dropped):
    orig = O.mlp_fp8

    def mutant(h, Xq, s_x, Wq, s_w, Wdq, s_wd, s_a, eps, bn):
        res = orig(h, Xq, 1.0 if dropped == "s_x" else s_x, Wq, s_w, Wdq, 1.0 if dropped == "s_wd" else s_wd,
                   s_a, eps, bn)
        if dropped == "s_a":   # a quantised at s_a but dequantised without it
            res = dict(res, Y=(res["Y"] - np.asarray(h, float)) / s_a + np.asarray(h, float))
        return res
    _plant(monkeypatch, "mlp_fp8", mutant)
    assert _fails(pins.test_mlp_fp8_power_of_two_scales_are_exact)


@pytest.mark.parametrize("dropped", ["s_x", "s_wd", "s_a"])
def test_mlp_nvfp4_dropped_tensor_scale_is_caught(monkeypatch, dropped):
    orig = O.mlp_nvfp4

    def mutant(h, Xq, Xsf, s_x, Wq, Wsf, s_w, Wdq, Wdsf, s_wd, s_a, eps, bn):
        with np.errstate(over="ignore"):   # without s_x, Z is 64x too large: sigmoid's exp overflows
            res = orig(h, Xq, Xsf, 1.0 if dropped == "s_x" else s_x, Wq, Wsf, s_w, Wdq, Wdsf,
                       1.0 if dropped == "s_wd" else s_wd, s_a, eps, bn)
        if dropped == "s_a":   # a quantised at s_a but dequantised without it
            res = dict(res, Y=(res["Y"] - np.asarray(h, float)) / s_a + np.asarray(h, float))
        return res
    _plant(monkeypatch, "mlp_nvfp4", mutant)
    assert _fails(fp4pins.test_mlp_nvfp4_power_of_two_scales_are_exact)


def test_qkv_rope_positions_without_the_sequence_wrap_are_caught(monkeypatch):
    # positions taken as the row index of the whole batch instead of the index within a sequence
    def mutant(h, g, W_qkv, eps, seq_len, n_rot_cols, head_dim, base):
        Z = O.linear(O.rmsnorm(h, g, eps), W_qkv)
        return dict(r=O.rms_scale(h, eps), Z=Z,
                    out=O.rope_rotate(Z, np.arange(Z.shape[0]), n_rot_cols, head_dim, base))
    _plant(monkeypatch, "qkv_rope", mutant)
    assert _fails(pins.test_qkv_rope_chain_is_norm_then_gemm_then_rotate)


def test_deferred_r_on_the_gate_half_only_is_caught(monkeypatch):
    def mutant(O_, R, W_o, g, W_gu, W_d, eps, bn):
        h = O.linear(O_, W_o) + np.asarray(R, float)
        P = O.partial_sumsq(h, bn)
        r = O.rms_scale_from_partials(P, h.shape[1], eps)
        Z = O.linear(h, O.fold_gain(W_gu, g))
        F = Z.shape[1] // 2
        Z[:, :F] *= r[:, None]             # r left off the up half
        G, U = Z[:, :F], Z[:, F:]
        a = O.swiglu(G, U)
        Y = O.linear(a, W_d) + h
        return dict(h=h, P=P, r=r, Z=Z, G=G, U=U, a=a, Y=Y)
    _plant(monkeypatch, "block_forward_deferred", mutant)
    assert _fails(pins.test_deferred_r_equals_naive)


def _nvfp4_bwd_variant(transform):
    """A copy of the oracle's NVFP4 MLP backward with one planted change applied by `transform`
    to the source of the function."""
    import inspect
    src = inspect.getsource(OC.mlp_nvfp4_backward)
    mutated = transform(src)
    assert mutated != src
    ns = dict(OC.__dict__)
    exec(mutated, ns)
    return ns["mlp_nvfp4_backward"]


def test_nvfp4_bwd_dy_quantised_along_the_wrong_axis_is_caught(monkeypatch):
    import tests.test_oracle_nvfp4_bwd as bwd
    bad = _nvfp4_bwd_variant(lambda s: s.replace("dW_d = Rc(dY, s_dy).T", "dW_d = Rr(dY, s_dy).T"))
    _plant(monkeypatch, "mlp_nvfp4_backward", bad)
    assert _fails(bwd.test_quantised_gradients_match_brute_force_blocks_along_each_contraction)


def test_nvfp4_bwd_e_quantised_along_the_wrong_axis_is_caught(monkeypatch):
    import tests.test_oracle_nvfp4_bwd as bwd
    bad = _nvfp4_bwd_variant(lambda s: s.replace("dW = Rc(e, s_e).T", "dW = Rr(e, s_e).T"))
    _plant(monkeypatch, "mlp_nvfp4_backward", bad)
    assert _fails(bwd.test_quantised_gradients_match_brute_force_blocks_along_each_contraction)


def test_nvfp4_bwd_dropped_rmsnorm_term_is_caught(monkeypatch):
    import tests.test_oracle_nvfp4_bwd as bwd
    bad = _nvfp4_bwd_variant(lambda s: s.replace("dh = t - c[:, None] * h + dY", "dh = t + dY"))
    _plant(monkeypatch, "mlp_nvfp4_backward", bad)
    assert _fails(bwd.test_unquantised_gradients_are_the_finite_differences)
