"""Error metrics shared by the parity tests.

The gate is the normalised max error max|got - ref| / max|ref| over a whole
tensor, and the same quantity per (b, h) slice (output magnitudes differ by
two orders of magnitude between heads with fast and slow decay, so a global
normalisation alone would hide errors in the fast heads).
Tolerances: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.
"""
from __future__ import annotations

import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def norm_err(got, ref) -> float:
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    scale = np.max(np.abs(ref))
    if scale == 0.0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / scale)


def per_head_err(got, ref) -> float:
    """Worst normalised error over the leading (B, H) slices."""
    got, ref = _np(got), _np(ref)
    B, H = ref.shape[:2]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            worst = max(worst, norm_err(got[b, h], ref[b, h]))
    return worst


def assert_close(got, ref, tol, what, per_head=True):
    e = norm_err(got, ref)
    assert np.all(np.isfinite(_np(got))), f"{what}: non-finite values"
    assert e <= tol, f"{what}: normalised error {e:.3e} > {tol:.1e}"
    if per_head and _np(ref).ndim >= 3:
        eh = per_head_err(got, ref)
        assert eh <= tol, f"{what}: per-head normalised error {eh:.3e} > {tol:.1e}"
    return e
