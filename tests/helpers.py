"""Shared test helpers: the error metrics and host<->device marshalling."""
import numpy as np
import torch

# (test id, tensor name, max relative error, max per-element relative error)
# of every comparison made through `checked`; printed at the end of the run.
PARITY_LOG = []


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


def max_elem_rel_err(got, ref) -> float:
    """max over elements of |got - ref| / (|ref| + 1e-6 max |ref|): the
    per-element figure, reported beside max_rel_err (not a bound: where a
    gradient entry is a near-cancelling sum, its own magnitude is far below
    the rounding of the terms it sums)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if g.size == 0:
        return 0.0
    if not np.all(np.isfinite(g)):
        return float("inf")
    floor = 1e-6 * np.max(np.abs(r))
    if floor == 0.0:
        return float(np.max(np.abs(g - r)))
    return float(np.max(np.abs(g - r) / (np.abs(r) + floor)))


def checked(name, got, ref, tag="") -> float:
    """max_rel_err of one output, with both error figures logged for the
    end-of-run parity report."""
    e = max_rel_err(got, ref)
    PARITY_LOG.append((tag, name, e, max_elem_rel_err(got, ref)))
    return e


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a tensor's values (bf16 values are exact in f64)."""
    return t.detach().to("cpu", torch.float64).numpy()


TOL_F32 = 1e-4    # fp32 inputs
TOL_BF16 = 2e-2   # bf16 inputs, fp32 accumulation
