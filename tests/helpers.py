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


def max_abs(got, ref):
    return float(np.max(np.abs(np64(got) - np64(ref)))) if np.size(ref) else 0.0


# Tolerances: relative Frobenius error per output tensor.
TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}
