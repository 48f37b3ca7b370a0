"""Storage roundings the method performs (oracle; test infrastructure only).

Every cast is a single round-to-nearest-even from the float64 value
([PR48792] §Tests: the builder rejects stochastic rounding, and §Out of scope:
stochastic rounding for a low-precision state is not part of the path).

NumPy's float64 -> float16 and float64 -> float32 conversions are single,
correctly rounded IEEE conversions (ties to even); bf16 is done here from the
float64 value by rounding the 53-bit significand to 8 bits (ties to even),
exponent range of fp32, overflow to inf.

Parity: pinned by tests on exact tie cases and representable values.
"""

import numpy as np

STORAGE_DTYPES = ("f64", "f32", "f16", "bf16")


def _round_bf16(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    m, e = np.frexp(xf)  # xf = m * 2**e, 0.5 <= |m| < 1
    # keep 8 significant bits: scale |m| to [128, 256), round half to even
    scaled = m * 256.0
    r = np.round(scaled)  # NumPy rounds half to even
    y = np.ldexp(r / 256.0, e)
    # bf16 max finite = (2 - 2^-7) * 2^127; values that round beyond it overflow
    y = np.where(np.abs(y) > (2.0 - 2.0 ** -7) * 2.0 ** 127, np.sign(y) * np.inf, y)
    # below the fp32 normal range bf16 is subnormal with step 2^-133
    tiny = np.abs(xf) < 2.0 ** -126
    if np.any(tiny):
        y[tiny] = np.round(xf[tiny] / 2.0 ** -133) * 2.0 ** -133
    out[finite] = y
    return out


def round_to(x, dtype):
    """Round float64 ``x`` to storage type ``dtype`` and return it as float64."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        return _round_bf16(x)
    raise ValueError(f"unknown storage dtype {dtype!r}")
