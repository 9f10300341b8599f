"""Comparison rules shared by the tests (no attention arithmetic here).

Tolerance: an output element passes when
    |gpu - oracle| <= 4 * ulp_bf16(max_v |oracle[row, :]|),
with ulp_bf16(x) = 2**(floor(log2 x) - 7) -- 4 bf16 ULP relative to the row's
largest magnitude, the gate the project's accuracy target states.  A row whose
oracle values are all zero must match exactly.
"""
from __future__ import annotations

import numpy as np

ULP_TOL = 4.0


def bits_to_f32(a) -> np.ndarray:
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    x = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    return np.where(x > 0, np.exp2(e - 7.0), 0.0)


def row_ulp_error(test, ref) -> np.ndarray:
    """Per-element error in units of bf16 ULP of the reference row's max |value|.

    ``test`` and ``ref`` are float arrays [..., n]; returns an array of the same
    shape (0 where both are exactly equal, inf where the row max is 0 and they
    differ)."""
    test = np.asarray(test, np.float64)
    ref = np.asarray(ref, np.float64)
    unit = ulp_bf16(np.max(np.abs(ref), axis=-1, keepdims=True))
    diff = np.abs(test - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(diff == 0, 0.0, diff / unit)
    return err


def assert_rows_close(test, ref, tol=ULP_TOL, what="output"):
    err = row_ulp_error(test, ref)
    assert np.all(np.isfinite(np.asarray(test, np.float64))), f"{what}: non-finite values"
    worst = float(np.max(err)) if err.size else 0.0
    assert worst <= tol, f"{what}: max error {worst:.3f} row-max bf16 ULP > {tol}"
    return err


def argmax_mismatch_ok(scores_row: np.ndarray, probs_row: np.ndarray, n: int, a_ref: int,
                       a_test: int) -> bool:
    """The argmax rule: equal, or the token the test picked has a reference bf16
    score within one bf16 ULP of the reference maximum, or a reference bf16
    probability tied at the maximum (the '<= 1-ULP coin flip' the source pages
    describe)."""
    if a_ref == a_test:
        return True
    if not (0 <= a_test < n):
        return False
    s = scores_row[:n].astype(np.float64)
    top = s.max()
    if s[a_test] >= top - float(ulp_bf16(np.array([top]))[0]):
        return True
    p = bits_to_f32(probs_row[:n])
    return bool(p[a_test] == p.max())
