"""Small helpers shared by the parity tests (no method arithmetic here)."""
import numpy as np
import torch


def np64(t):
    """Tensor (any device / dtype) -> float64 numpy array with the same values."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(got, ref):
    got, ref = np64(got), np64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def bf16_step(x):
    """One bf16 rounding step (unit in the last place) at magnitude |x|."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    return np.where(x > 0, np.exp2(e - 7), 0.0)


def rel_rows(got, ref, row, bf16_outputs=False):
    """Largest relative error of any row of `row` consecutive elements (one
    head vector, one model-width row, one vocabulary row): ||g - r|| / ||r||
    per row, the absolute error where a reference row is exactly zero.

    bf16_outputs: both sides store the row in bf16, each rounding its own
    (float32 / float64) value, and two roundings of nearly the same value can
    land one bf16 step apart.  One such step of the row's largest element is
    subtracted from the row's error before it is compared: a single rounding
    flip of a dominant element is allowed, a wrong row is not."""
    got, ref = np64(got).reshape(-1, row), np64(ref).reshape(-1, row)
    if ref.shape[0] == 0:
        return 0.0
    num = np.linalg.norm(got - ref, axis=1)
    if bf16_outputs:
        num = np.maximum(0.0, num - bf16_step(np.max(np.abs(ref), axis=1)))
    den = np.linalg.norm(ref, axis=1)
    return float(np.max(num / np.where(den > 0, den, 1.0)))


def max_abs(got, ref):
    return float(np.max(np.abs(np64(got) - np64(ref)))) if np.size(ref) else 0.0


# Tolerances: relative error per output tensor (Frobenius) and per output row.
TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}


def assert_close(got, ref, tol, row, what=""):
    """Both bounds at `tol` (a dtype key of TOL or a number; a bf16 dtype also
    means bf16-stored outputs): the relative Frobenius error of the whole
    output, and the relative error of its worst row of `row` elements (less
    one bf16 step of the row's largest element for bf16 outputs, see
    rel_rows)."""
    bf16 = tol is torch.bfloat16 or (not isinstance(tol, torch.dtype) and getattr(got, "dtype", None) == torch.bfloat16)
    tol = TOL[tol] if isinstance(tol, torch.dtype) else float(tol)
    f, r = rel_fro(got, ref), rel_rows(got, ref, row, bf16_outputs=bf16)
    r_plain = rel_rows(got, ref, row)
    print("%s: rel %.2e, worst row %.2e (%.2e before the rounding-step allowance), max abs %.2e"
          % (what, f, r, r_plain, max_abs(got, ref)))
    assert f <= tol and r <= tol, (what, "rel", f, "worst row", r, "max abs", max_abs(got, ref))
    return f, r
