"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""
import numpy as np
import torch


def to64(t):
    """bf16/fp32 torch tensor (any device) -> float64 numpy, exactly."""
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(name, got, want, atol, rtol, extra=None):
    """|got - want| <= atol + rtol |want| (+ an element-wise ``extra`` allowance)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - want)
    tol = atol + rtol * np.abs(want)
    if extra is not None:
        tol = tol + np.asarray(extra, dtype=np.float64)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside atol={atol} rtol={rtol}; "
                             f"worst at {i}: got {got[i]!r} want {want[i]!r} (max abs err {err.max():.3g})")
