"""Pins of the oracle's residual add + RMS normalisation against what the
mathematics fixes ("Inference Engineering VII.07: Kernel and Operator
Fusion" page, sections 4-5: h = x + residual, out = h * rsqrt(mean(h^2) +
eps) * weight, both returned).

Each pin is a closed form, an invariant or a library routine, chosen so that
a plausible slip in the oracle fails one of them: eps dropped or added
outside the root, sum instead of mean, the weight or the residual left out,
sqrt instead of its reciprocal, a row mixed into another."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_40_gb300 import synth


def bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def test_new_residual_is_the_exact_sum():
    x, r, w = synth.norm_inputs_shape(11, 5, 96)
    _, h = oracle.add_rms_norm(x, r, w, 1e-6)
    assert np.array_equal(h, f64(x) + f64(r))


def test_constant_row_closed_form():
    # h_i = c for all i: mean(h^2) = c^2, so out_i = c / sqrt(c^2 + eps) * w_i
    D = 64
    w = bf16(np.linspace(0.5, 2.0, D))
    for c_x, c_r, eps in [(1.5, 0.25, 1e-6), (-3.0, 0.5, 0.1), (0.0078125, 0.0, 1e-4)]:
        x = np.tile(bf16([c_x]), (2, D))
        r = np.tile(bf16([c_r]), (2, D))
        out, _ = oracle.add_rms_norm(x, r, w, eps)
        c = c_x + c_r
        want = c / np.sqrt(c * c + eps) * f64(w)
        np.testing.assert_allclose(out, np.tile(want, (2, 1)), rtol=1e-14, atol=0)


def test_unit_rms_without_eps():
    # eps = 0: (out / w) has mean square exactly 1 in every row
    x, r, w = synth.norm_inputs_shape(12, 7, 200)
    out, _ = oracle.add_rms_norm(x, r, w, 0.0)
    ms = np.mean((out / f64(w)) ** 2, axis=1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-13)


def test_scale_invariance_without_eps():
    # eps = 0: scaling a row by 2 (exact in bf16) leaves out unchanged
    x, r, w = synth.norm_inputs_shape(13, 3, 128)
    x2 = bf16(2.0 * synth.bf16_bits_to_f32(x))
    r2 = bf16(2.0 * synth.bf16_bits_to_f32(r))
    a, _ = oracle.add_rms_norm(x, r, w, 0.0)
    b, _ = oracle.add_rms_norm(x2, r2, w, 0.0)
    np.testing.assert_allclose(b, a, rtol=1e-14, atol=1e-300)


def test_one_hot_row():
    # h = a e_k: mean(h^2) = a^2 / D, out_k = a / sqrt(a^2 / D + eps) w_k, rest 0
    D, k, a, eps = 256, 37, 4.0, 1e-3
    x = np.zeros((1, D), np.uint16)
    x[0, k] = bf16([a])[0]
    r = np.zeros((1, D), np.uint16)
    w = bf16(np.full(D, 1.25))
    out, _ = oracle.add_rms_norm(x, r, w, eps)
    want = np.zeros(D)
    want[k] = a / np.sqrt(a * a / D + eps) * 1.25
    np.testing.assert_allclose(out[0], want, rtol=1e-14, atol=0)


def test_zero_row_gives_zero():
    x = np.zeros((2, 32), np.uint16)
    w = bf16(np.ones(32))
    out, h = oracle.add_rms_norm(x, x.copy(), w, 1e-6)
    assert not out.any() and not h.any()


def test_rows_are_independent():
    x, r, w = synth.norm_inputs_shape(14, 6, 80)
    full, _ = oracle.add_rms_norm(x, r, w, 1e-6)
    for i in (0, 3, 5):
        one, _ = oracle.add_rms_norm(x[i:i + 1], r[i:i + 1], w, 1e-6)
        assert np.array_equal(one[0], full[i])


@pytest.mark.skipif(not hasattr(torch.nn.functional, "rms_norm"), reason="torch without rms_norm")
def test_matches_torch_rms_norm_fp64():
    # library special case: torch's RMSNorm of the summed row, in fp64 on CPU
    x, r, w = synth.norm_inputs_shape(15, 9, 512)
    out, h = oracle.add_rms_norm(x, r, w, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(f64(x) + f64(r)), (512,),
                                       torch.from_numpy(f64(w)), 1e-6).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_rejects_bad_arguments():
    x = np.zeros((1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.add_rms_norm(x, x, np.zeros(8, np.uint16), -1.0)
    with pytest.raises(ValueError):
        oracle.add_rms_norm(x, x, np.zeros(7, np.uint16), 1e-6)
