"""Scalar numerics of the oracle: storage rounding, sanitize, HDR transfer.

Readings (the helpers are imported by the pages but their bodies are absent):

* storage rounding - IEEE round-to-nearest-even to fp16 (subnormals kept,
  overflow to +-Inf) or fp32, applied once to the exact (fp64) value;
* sanitize(v, lo, hi) - NaN becomes 0, then v < lo gives lo and v > hi gives
  hi, component-wise (so +-Inf clamp to the bounds and -0.0 passes through);
* HDR 'log' transfer - F(x) = log2(1 + x), F^-1(y) = 2^y - 1.
"""

import numpy as np

FLT_MAX = np.float32(np.finfo(np.float32).max)


def round_storage(x, precision):
    """Round an array (any float dtype) once to the storage type.

    fp16 storage of activations and of fp16 weights ("nativeUNet.ts",
    storeExpression / packConvTensors); fp32 otherwise.
    """
    if precision == "fp16":
        return np.asarray(x, dtype=np.float64).astype(np.float16)
    if precision == "fp32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    raise ValueError(precision)


def sanitize(v, lo, hi):
    """sanitize(v, lo, hi) on float32 data ("denoise.ts", inputShader and
    outputShader call it; reading: NaN -> 0, then clamp by comparison)."""
    v = np.asarray(v, dtype=np.float32)
    lo = np.float32(lo)
    hi = np.float32(hi)
    out = np.where(np.isnan(v), np.float32(0.0), v)
    out = np.where(out < lo, lo, out)
    out = np.where(out > hi, hi, out)
    return out.astype(np.float32)


def hdr_forward_exact(x):
    """F(x) = log2(1 + x) in float64 for float32 inputs x >= 0."""
    x = np.asarray(x, dtype=np.float64)
    return np.log1p(x) / np.log(2.0)


def hdr_inverse_exact(y):
    """F^-1(y) = 2^y - 1 in float64 for float32 inputs y >= 0.

    2^y - 1 is taken as written for y >= 1 (2^y >= 2, so the subtraction
    loses at most one bit); below 1, where it cancels, as expm1(y ln 2)."""
    y = np.asarray(y, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.where(y < 1.0, np.expm1(y * np.log(2.0)), np.exp2(y) - 1.0)
