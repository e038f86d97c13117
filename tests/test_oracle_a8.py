"""Pins of the oracle's 8-bit activation variant (radiance_escha.py,
escha_linear_into: escha_pre_quant writes uint8 A [M][IC] with a float32 row
scale As from a row amax).  The codes are checked against the rounding bound
and the row maximum, the product against a dense numpy formulation on the
independently pinned decoded weights and scipy's Hadamard matrix, and the
whole against exact scaling and zero identities."""
import numpy as np
import pytest
import scipy.linalg

import oracle
import synthetic as syn


def _case(seed, M=5, IC=256, OC=384, K=3):
    return syn.linear_case(seed, M, IC, OC, K)


def test_codes_round_to_nearest_and_hit_the_row_maximum():
    x, sh = _case(1)
    _, A, As = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, nblk=0)
    u = oracle.pretransform_f64(x, sh.s_in, sh.rin)
    q = A.astype(np.int64) - 128
    assert np.all(np.abs(q) <= 127)
    np.testing.assert_allclose(As, np.abs(u).max(axis=1) / 127, rtol=1e-15)
    # every code is within half a step of its value, and the largest magnitude is 127
    assert np.all(np.abs(q * As[:, None] - u) <= As[:, None] / 2 * (1 + 1e-12))
    assert np.all(np.abs(q).max(axis=1) == 127)


def test_product_matches_dense_formulation():
    x, sh = _case(2)
    y, A, As = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    W = oracle.reconstruct(sh.code, sh.K).view(np.float16).astype(np.float64)
    uq = (A.astype(np.float64) - 128) * As[:, None]
    v = uq @ W
    H = scipy.linalg.hadamard(128) / np.sqrt(128)
    hv = (v.reshape(v.shape[0], -1, 128) @ H).reshape(v.shape)
    ref = hv * sh.rout.view(np.float16).astype(np.float64) * sh.s_out.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_scaling_the_input_scales_the_output_only():
    x, sh = _case(3)
    y1, A1, s1 = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    x2 = (x.astype(np.uint32) + (1 << 7)).astype(np.uint16)   # bf16 exponent + 1: x * 2 exactly
    y2, A2, s2 = oracle.linear_a8_f64(x2, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert np.array_equal(A1, A2)
    np.testing.assert_array_equal(s2, 2 * s1)
    np.testing.assert_array_equal(y2, 2 * y1)


def test_zero_rows():
    x, sh = _case(4)
    x[1] = 0
    y, A, As = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert As[1] == 0 and np.all(A[1] == 128) and np.all(y[1] == 0)


def test_close_to_the_unquantized_layer():
    # 8-bit activations: each code is off by at most half a step, so the result stays
    # within a few percent of the layer on the exact activations
    x, sh = _case(5, M=8, IC=1024, OC=512)
    ya8, _, _ = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    y = oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    rel = np.sqrt(np.mean((ya8 - y) ** 2, axis=1)) / np.sqrt(np.mean(y ** 2, axis=1))
    assert np.all(rel < 0.03)
