"""Shared test helpers: error metric and dtype conversions (no method arithmetic)."""

import numpy as np


def rel_err(x, y, nd=1):
    """Max relative error of ``x`` against reference ``y``.

    Per element |x - y| / max(|y|, rms(y over its head vector or matrix)), the
    RMS guarding elements of ``y`` near zero; ``nd`` trailing axes form one
    head's vector (1) or matrix (2).  Returns the maximum over all elements.
    """
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if x.size == 0:
        return 0.0
    axes = tuple(range(-nd, 0))
    rms = np.sqrt(np.mean(y * y, axis=axes, keepdims=True))
    denom = np.maximum(np.maximum(np.abs(y), rms), 1e-30)
    err = np.abs(x - y) / denom
    if np.any(np.isnan(err)):
        return float("inf")
    return float(np.max(err))


def f64(a):
    """NumPy float64 copy of a NumPy array or a (CPU/GPU) torch tensor."""
    try:
        import torch

        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)
