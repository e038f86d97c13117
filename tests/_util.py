"""Shared helpers for the GPU parity tests (host-side marshalling and the
per-row tolerance).

Tolerance: |y - y_ref| <= 2e-2 * rms(y_ref row) + ulp_bf16(y_ref) / 2 for every
element, y_ref the exact (fp64) oracle value.  The 2e-2 * rms term bounds the
arithmetic (fp16 operands, fp32 accumulation); the half-ulp term is the bf16
storage of the result itself, which for an element beyond ~5 rms exceeds the
first term on its own (bf16 keeps 8 significant bits).
"""
import numpy as np
import torch

TOL = 2e-2


def dev(a, dtype, device="cuda"):
    """numpy bits -> device tensor of the given dtype (same bytes)."""
    a = np.ascontiguousarray(a)
    view = {torch.bfloat16: np.int16, torch.float16: np.int16}.get(dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a).to(device).view(dtype)


def bits(t):
    """16-bit device tensor -> numpy uint16 bits."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(v):
    """Half the spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def row_err_ratio(got, ref):
    """Per-row max|got - ref| / rms(ref) (the raw statistic, bf16 storage included)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1))
    err = np.max(np.abs(got - ref), axis=-1)
    return err / np.maximum(rms, 1e-30)


def excess_ratio(got, ref):
    """Per-row max over elements of (|got - ref| - ulp_bf16(ref)/2) / rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    ex = (np.abs(got - ref) - half_ulp_bf16(ref)) / np.maximum(rms, 1e-30)
    return np.max(ex, axis=-1)


def assert_rows_close(got, ref, tol=TOL):
    assert np.all(np.isfinite(got)), "non-finite output"
    r = excess_ratio(got, ref)
    assert np.all(r <= tol), (f"row tolerance exceeded: worst (|err| - ulp/2)/rms = {r.max():.3e} (> {tol}); "
                              f"raw max|err|/rms = {row_err_ratio(got, ref).max():.3e}")
    return r.max()
