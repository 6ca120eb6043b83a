"""Tolerances shared by the parity tests.

fp32 state / outputs / records against the fp64 oracle:
    |gpu - ref| <= ATOL + RTOL * |ref|,  ATOL = RTOL = 1e-4.
bf16 state after the commit's single rounding:
    |gpu - ref| <= bf16_ulp(ref) + BF16_FLOOR
where bf16_ulp(x) is the spacing of the bf16 grid at |x| and BF16_FLOOR
absorbs the fp32 rounding of the fold before the one bf16 rounding (the
fold's own error is bounded by ~2 * n * 2^-24 * max|term|, well below
1e-6 for states of magnitude <= 4 and n <= 16 tokens).
"""
import math

import numpy as np

ATOL = 1e-4
RTOL = 1e-4
BF16_FLOOR = 1e-6


def bf16_ulp(x):
    """Spacing of the bf16 grid (8 significant bits) at |x|, elementwise."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    e = np.where(x > 0, np.maximum(e, -126.0), -126.0)
    return np.exp2(e - 7.0)


def check_close(gpu, ref, what, atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside tol; worst at {i}: "
            f"gpu={gpu[i]!r} ref={ref[i]!r} err={err[i]:.3e}")
    return float(err.max()) if err.size else 0.0


def check_bf16(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = bf16_ulp(ref) + BF16_FLOOR
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} beyond 1 bf16 ulp; worst at {i}: "
            f"gpu={gpu[i]!r} ref={ref[i]!r}")
    return float((err / bf16_ulp(ref)).max()) if err.size else 0.0


def log2_int(x):
    return int(math.floor(math.log2(abs(x))))
