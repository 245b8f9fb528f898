"""Shared test helpers: the error metric and host<->device marshalling."""
import numpy as np
import torch


def max_rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| over one output tensor (the reading of
    "max relative error" used for every parity bound)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if not np.all(np.isfinite(g)):
        return float("inf")
    denom = np.max(np.abs(r))
    if denom == 0.0:
        return float(np.max(np.abs(g - r)))
    return float(np.max(np.abs(g - r)) / denom)


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a tensor's values (bf16 values are exact in f64)."""
    return t.detach().to("cpu", torch.float64).numpy()


TOL_F32 = 1e-4    # fp32 inputs
TOL_BF16 = 2e-2   # bf16 inputs, fp32 accumulation
