"""Output comparison used by every parity test.

The bar for bf16 outputs: for every element
``|y - r| / max(|r|, 1e-2 * rms(r)) <= 8e-3`` (max relative error, with a floor
so that results that cancel to about zero do not divide by zero), and
``|y - r| <= ulp_bf16(r)`` for at least 99.9% of the elements, where ``r`` is
the oracle's fp32 result and ``ulp_bf16(r) = 2^(floor(log2|r|) - 7)``.
"""
import numpy as np

REL_TOL = 8e-3
ULP_FRACTION = 0.999


def bf16_bits_to_f64(bits):
    return (np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def ulp_bf16(r):
    a = np.abs(np.asarray(r, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    return np.exp2(e - 7)


def check_bf16_output(y_bits, r, what=""):
    y = bf16_bits_to_f64(y_bits)
    r = np.asarray(r, dtype=np.float64)
    assert y.shape == r.shape, (y.shape, r.shape)
    if r.size == 0:
        return
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    rms = np.sqrt(np.mean(r * r))
    floor = max(1e-2 * rms, 1e-30)
    err = np.abs(y - r)
    rel = err / np.maximum(np.abs(r), floor)
    worst = np.unravel_index(np.argmax(rel), rel.shape)
    assert rel.max() <= REL_TOL, (
        f"{what}: max rel err {rel.max():.3e} at {worst}: y={y[worst]!r} r={r[worst]!r}")
    within = np.mean(err <= ulp_bf16(r))
    assert within >= ULP_FRACTION, f"{what}: only {within:.5f} of elements within 1 bf16 ulp"
