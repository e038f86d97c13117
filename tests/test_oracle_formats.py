"""Pins the oracle's hand-written fp16 / bf16 conversions to numpy and torch."""
import numpy as np
import torch

import oracle


def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(b) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(b) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def _f16_round_cases(g):
    # random normals over the whole fp16 range, subnormals, exact ties, overflow edge
    v = np.concatenate([
        g.standard_normal(4000) * 10.0 ** g.uniform(-8, 5, 4000),
        g.uniform(0, 2 ** -14, 2000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2 ** -25, 2 ** -24,
                  3 * 2 ** -26, 2 ** -25 * 1.0000001]),
    ])
    # exact midpoints between consecutive fp16 values (ties to even)
    h = np.arange(0, 0x7C00, 3, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = (np.arange(0, 0x7C00, 3, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    ties = (h + nxt) / 2.0
    return np.concatenate([v, ties, -ties])


def test_f16_encode_matches_numpy():
    g = np.random.default_rng(0)
    v = _f16_round_cases(g)
    ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_from_f64(x) for x in v], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_torch_on_f32_exact_values():
    # torch rounds float32 -> bf16 with one rounding; restrict to doubles that are
    # exact float32 values (including exact bf16 ties) so both sides round once.
    g = np.random.default_rng(1)
    f = (g.standard_normal(20000) * 10.0 ** g.uniform(-30, 30, 20000)).astype(np.float32)
    lo = np.arange(0, 0x7F7F, 5, dtype=np.uint32)
    ties = ((lo << 16) | 0x8000).astype(np.uint32).view(np.float32)
    f = np.concatenate([f, ties, -ties, np.float32([0, -0.0, 3.4e38, -3.4e38, 1e-40])])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_f64(float(x)) for x in f], np.uint16)
    assert np.array_equal(got, ref)
