"""Shared helpers for the GPU parity tests (host-side marshalling and the
per-row tolerance max|y - y_ref| <= 2e-2 * rms(y_ref))."""
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


def row_err_ratio(got, ref):
    """Per-row max|got - ref| / rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1))
    err = np.max(np.abs(got - ref), axis=-1)
    return err / np.maximum(rms, 1e-30)


def assert_rows_close(got, ref, tol=TOL):
    r = row_err_ratio(got, ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    assert np.all(r <= tol), f"row tolerance exceeded: worst max|err|/rms = {r.max():.3e} (> {tol})"
    return r.max()
