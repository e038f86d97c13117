"""Pins of the oracle's int8 output head (vllm-quantpack exl3/embedding.py,
Exl3EmbeddingMethod.apply: the weight is the int8 table times its per-row scale,
and the head is x @ weight^T).  The oracle's plain loop is checked against
numpy's matrix product, against the (independently pinned) int8 gather through
one-hot inputs, and against exact zero / scaling identities."""
import numpy as np
import pytest

import oracle
import synthetic as syn

pytestmark = pytest.mark.filterwarnings("ignore")


def _case(seed, M, V, H):
    q, s, _ = syn.embedding(seed, V=V, H=H, N=1)
    g = syn.rng(seed + 1)
    x = syn.normal_bf16(g, M, H)
    return x, q, s


def test_matches_numpy_matrix_product():
    x, q, s = _case(1, 5, 300, 256)
    xf = np.array([oracle.bf16_to_f64(int(b)) for b in x.ravel()]).reshape(x.shape)
    sf = s.view(np.float16).astype(np.float64)
    ref = (xf @ q.astype(np.float64).T) * sf[None, :]
    got = oracle.lm_head_f64(x, q, s)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_vocabulary_window_equals_full_head():
    x, q, s = _case(2, 3, 200, 128)
    full = oracle.lm_head_f64(x, q, s)
    part = oracle.lm_head_f64(x, q, s, v0=37, nv=90)
    assert np.array_equal(part, full[:, 37:127])


def test_one_hot_inputs_give_the_gathered_rows():
    # x = e_j selects column j of the weight: s[v] * q[v][j] for every row v, which
    # the gather oracle produces (rounded once to bf16) for ids = 0..V-1
    V, H = 96, 64
    _, q, s = _case(3, 1, V, H)
    x = np.zeros((H, H), np.uint16)
    x[np.arange(H), np.arange(H)] = 0x3F80          # bf16 1.0
    head = oracle.lm_head_f64(x, q, s)              # [H][V]: row j = column j of w
    rows, bad = oracle.gather(q, s, np.arange(V, dtype=np.int32))
    assert bad == 0
    assert np.array_equal(oracle.bf16_bits_from_f64_array(head.T), rows)


def test_zero_input_and_scale_linearity():
    x, q, s = _case(4, 4, 120, 128)
    assert np.array_equal(oracle.lm_head_f64(np.zeros_like(x), q, s), np.zeros((4, 120)))
    s2 = (s.view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(oracle.lm_head_f64(x, q, s2), 2 * oracle.lm_head_f64(x, q, s))
