"""Element-by-element parity of CUDA bf16 outputs against the oracle.

Tolerance (the stated bar for floating-point outputs): every element obeys
    |gpu - oracle| <= 2^-7 * |oracle| + 1e-6,
no element is more than one bf16 step (ulp) away from the oracle's rounded
value unless it is also within 1e-6 of it (values next to zero, where a
rotation's fp32 cancellation legitimately moves more than one step), and at
most 0.1% of all elements are exactly one step away.  Steps are counted on
the sign-magnitude order of bf16 bit patterns, so +0 and -0 are 0 apart.
"""
from __future__ import annotations

import numpy as np

from tests.exact import bits_to_f64, ulp_distance_bf16

ABS_FLOOR = 1e-6
REL_BOUND = 2.0**-7
MAX_ONE_ULP_FRACTION = 1e-3


def parity_report(gpu_bits, ref_bits, abs_floor=None) -> dict:
    """`abs_floor` (scalar or per-element array) replaces the 1e-6 absolute
    floor where an operation's own fp32 error bound is larger (LayerNorm rows
    with a large mean: the centring x - mean carries |mean| * 2^-24)."""
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16).ravel()
    ref_bits = np.asarray(ref_bits, dtype=np.uint16).ravel()
    assert gpu_bits.shape == ref_bits.shape
    floor = ABS_FLOOR if abs_floor is None else np.maximum(
        ABS_FLOOR, np.broadcast_to(np.asarray(abs_floor, dtype=np.float64), gpu_bits.shape))
    g = bits_to_f64(gpu_bits)
    r = bits_to_f64(ref_bits)
    diff = np.abs(g - r)
    ulp = ulp_distance_bf16(gpu_bits, ref_bits)
    finite = np.isfinite(g) & np.isfinite(r)
    over_bound = ~(diff <= REL_BOUND * np.abs(r) + floor) | ~finite
    multi_ulp = (ulp > 1) & (diff > floor)
    bad = over_bound | multi_ulp
    n = max(1, gpu_bits.size)
    return {
        "n": int(gpu_bits.size),
        "bad": int(bad.sum()),
        "one_ulp": int((ulp == 1).sum()),
        "one_ulp_frac": float((ulp == 1).sum()) / n,
        "near_zero_multi_ulp": int(((ulp > 1) & (diff <= floor)).sum()),
        "exact": int((ulp == 0).sum()),
        "max_ulp": int(ulp.max()) if ulp.size else 0,
        "first_bad": (np.flatnonzero(bad)[:8].tolist()),
    }


def assert_parity(gpu_bits, ref_bits, what: str = "", abs_floor=None,
                  max_one_ulp_frac: float = MAX_ONE_ULP_FRACTION) -> dict:
    rep = parity_report(gpu_bits, ref_bits, abs_floor)
    assert rep["bad"] == 0, f"{what}: {rep['bad']} elements outside tolerance: {rep}"
    assert rep["one_ulp_frac"] <= max_one_ulp_frac, \
        f"{what}: {rep['one_ulp_frac']:.5%} elements one bf16 step off (> {max_one_ulp_frac:.2%}): {rep}"
    return rep
