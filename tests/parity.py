"""Error metrics and tolerances for comparing the CUDA path with the oracle.

* fp32 inputs: relative Frobenius error ||X - X_ref||_F / ||X_ref||_F <= 1e-5,
  over the whole tensor, for X in {O, S_final}.
* bf16 inputs (fp32 accumulation): per-row relative error
  ||x_r - x_ref,r||_2 / max(||x_ref,r||_2, f * RMS row norm) <= 2e-2 for
  every row, where a row is one d_v-vector (a token of O, a row of S), and
  f = 1e-6 unless a test sets the floor: rounding bf16 operands errs relative
  to the terms a row sums, so where those cancel (identity phi, whose scores
  take both signs) a test may hold a row to a floor of the typical row's norm.
"""
from __future__ import annotations

import numpy as np

TOL_F32_FROB = 1e-5
TOL_BF16_ROW = 2e-2


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_frobenius(x, ref) -> float:
    x, ref = _np(x), _np(ref)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def max_row_rel(x, ref, row_floor: float = 1e-6) -> float:
    x, ref = _np(x), _np(ref)
    if ref.size == 0:
        return 0.0
    xr = x.reshape(-1, x.shape[-1])
    rr = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(rr, axis=1)
    rms = float(np.sqrt(np.mean(rn ** 2)))
    den = np.maximum(rn, row_floor * rms if rms > 0 else 1e-30)
    return float(np.max(np.linalg.norm(xr - rr, axis=1) / den))


def check(x, ref, dtype: str, what: str, row_floor: float = 1e-6):
    """Assert the tolerance for the input dtype ("f32" | "bf16"); row_floor is
    the bf16 check's floor of a row's norm, as a fraction of the RMS row norm."""
    if dtype == "f32":
        e = rel_frobenius(x, ref)
        assert e <= TOL_F32_FROB, f"{what}: relative Frobenius error {e:.3e} > {TOL_F32_FROB}"
    else:
        e = max_row_rel(x, ref, row_floor)
        assert e <= TOL_BF16_ROW, f"{what}: max per-row relative error {e:.3e} > {TOL_BF16_ROW}"
    return e
