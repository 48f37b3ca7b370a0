"""Storage roundings the method performs (oracle; test infrastructure only).

Every cast is a single round-to-nearest-even from the float64 value
([PR48792] §Tests: the builder rejects stochastic rounding, and §Out of scope:
stochastic rounding for a low-precision state is not part of the path).

NumPy's float64 -> float16 and float64 -> float32 conversions are single,
correctly rounded IEEE conversions (ties to even); bf16 is done here from the
float64 value by rounding the 53-bit significand to 8 bits (ties to even),
exponent range of fp32, overflow to inf; E4M3 likewise to 4 significant bits
with its own exponent range and saturation at 448.

Parity: pinned by tests on exact tie cases and representable values.
"""

import numpy as np

STORAGE_DTYPES = ("f64", "f32", "f16", "bf16", "e4m3")

# FP8 E4M3 in the OCP "fn" encoding: exponent bias 7, 3 mantissa bits, no
# infinities; largest finite value 1.75 * 2^8 = 448, smallest normal 2^-6,
# subnormals k * 2^-9 (k = 1 .. 7)
E4M3_MAX = 448.0


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


def _round_e4m3(x):
    """Round to E4M3, nearest even, saturating: a value whose rounding lies
    beyond the largest finite value becomes +-448 (the saturating conversion
    the decode kernel uses; the format has no infinity)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    m, e = np.frexp(xf)  # xf = m * 2**e, 0.5 <= |m| < 1
    # normal numbers keep 4 significant bits (1 implicit + 3)
    y = np.ldexp(np.round(m * 16.0) / 16.0, e)
    # below 2^-6 the grid is the subnormal step 2^-9
    tiny = np.abs(xf) < 2.0 ** -6
    if np.any(tiny):
        y[tiny] = np.round(xf[tiny] / 2.0 ** -9) * 2.0 ** -9
    out[finite] = np.clip(y, -E4M3_MAX, E4M3_MAX)
    return out


def row_scale_exponent(x):
    """Exponent e of the power-of-two scale of each row (last axis) of an E4M3
    read copy: the smallest integer with max|row| <= 448 * 2^e (0 for a row of
    zeros).  Exact integer arithmetic on the row maximum."""
    amax = np.max(np.abs(np.asarray(x, dtype=np.float64)), axis=-1)
    m, k = np.frexp(amax)  # amax = m * 2**k, 0.5 <= m < 1;  448 = 0.875 * 2**9
    e = np.where(m <= 0.875, k - 9, k - 8)
    return np.where(amax > 0, e, 0).astype(np.int64)


def round_rows_scaled(x):
    """E4M3 read copy of a matrix: each row (last axis) is divided by its
    power-of-two scale 2^e (``row_scale_exponent``), rounded to E4M3 (nearest
    even) and multiplied back.  The division and the multiplication are
    exact, so the copy is one rounding of each element on the row's grid."""
    x = np.asarray(x, dtype=np.float64)
    e = row_scale_exponent(x)[..., None]
    return np.ldexp(_round_e4m3(np.ldexp(x, -e)), e)


def round_read_copy(x, dtype):
    """The read copy of a two-precision checkpoint ([Ghana] §The precision
    argument): one round-to-nearest-even cast of the unrounded state to fp16
    or bf16, or to E4M3 on a power-of-two scale per state row."""
    if dtype == "e4m3":
        return round_rows_scaled(x)
    return round_to(x, dtype)


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
    if dtype == "e4m3":
        return _round_e4m3(x)
    raise ValueError(f"unknown storage dtype {dtype!r}")
