"""Element-by-element parity of CUDA 16-bit outputs against the oracle.

Tolerance for bf16 (the stated bar for floating-point outputs): every element
obeys
    |gpu - oracle| <= 2^-7 * |oracle| + 1e-6,
no element is more than one bf16 step (ulp) away from the oracle's rounded
value unless it is also within 1e-6 of it (values next to zero, where a
rotation's fp32 cancellation legitimately moves more than one step), and at
most 0.1% of all elements are exactly one step away.  Steps are counted on
the sign-magnitude order of the bit patterns, so +0 and -0 are 0 apart.
Identical bit patterns (infinities included) always agree.

fp16 outputs carry the same fp32 arithmetic to a format with 3 more
significand bits.  An output moves by one step only when the kernel's
relative error eps_k straddles a rounding midpoint; for a value with relative
step u that happens with probability about 2 * eps_k / u.  bf16 has
u > 2^-8, so the 0.1% budget allows eps_k up to about 2^-19; fp16 has
u > 2^-11, so the same eps_k gives 8 times the fraction: the fp16 budget is
2^-7 (0.78%) one-step elements, and each element within one fp16 step
(2^-10 relative) of the oracle.

The fraction budget is a statement about large populations.  On small tests
built from degenerate rows it can be exceeded by correct fp32 arithmetic:
bf16 inputs have 128 mantissas per binade, so when a row's fp32 scale lands
within its rounding error of a midpoint for one mantissa, every element
sharing that mantissa (about N/128 of the row) moves together.  Such tests
pass `exact` (the unrounded oracle values) instead: then every one-step
element must lie within EXACT_REL (the kernels' fp32 error bound, 2^-20
relative, plus the absolute floor) of a rounding midpoint of the format,
which is stricter than the fraction budget for every other element.
"""
from __future__ import annotations

import numpy as np

from tests.exact import bits_to_f64, f16_bits_to_f64, ulp_distance_bf16

ABS_FLOOR = 1e-6
REL_BOUND = 2.0**-7
MAX_ONE_ULP_FRACTION = 1e-3
REL_BOUND_F16 = 2.0**-10
MAX_ONE_ULP_FRACTION_F16 = 2.0**-7
EXACT_REL = 2.0**-20


def near_midpoint(y_exact, fmt: str = "bf16", rel: float = EXACT_REL,
                  abs_floor: float = ABS_FLOOR) -> np.ndarray:
    """Whether each unrounded value lies within rel * |y| + abs_floor of a
    rounding midpoint of the format (the points where one fp32 rounding can
    move the result to the neighbouring 16-bit value)."""
    y = np.abs(np.asarray(y_exact, dtype=np.float64)).ravel()
    sig = 11 if fmt == "f16" else 8          # significant bits
    qmin = 2.0**-24 if fmt == "f16" else 2.0**-133
    _, e = np.frexp(np.where(y > 0, y, 1.0))  # y = f * 2^e, f in [0.5, 1)
    q = np.maximum(np.ldexp(1.0, e - sig), qmin)
    mid = (np.floor(y / q) + 0.5) * q
    return (np.abs(y - mid) <= rel * y + abs_floor) & (y > 0)


def parity_report(gpu_bits, ref_bits, abs_floor=None, fmt: str = "bf16", exact=None) -> dict:
    """`abs_floor` (scalar or per-element array) replaces the 1e-6 absolute
    floor where an operation's own fp32 error bound is larger (LayerNorm rows
    with a large mean: the centring x - mean carries |mean| * 2^-24)."""
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16).ravel()
    ref_bits = np.asarray(ref_bits, dtype=np.uint16).ravel()
    assert gpu_bits.shape == ref_bits.shape
    floor = ABS_FLOOR if abs_floor is None else np.maximum(
        ABS_FLOOR, np.broadcast_to(np.asarray(abs_floor, dtype=np.float64), gpu_bits.shape))
    decode = f16_bits_to_f64 if fmt == "f16" else bits_to_f64
    rel = REL_BOUND_F16 if fmt == "f16" else REL_BOUND
    g = decode(gpu_bits)
    r = decode(ref_bits)
    with np.errstate(invalid="ignore"):
        diff = np.abs(g - r)
    ulp = ulp_distance_bf16(gpu_bits, ref_bits)  # sign-magnitude order: any 16-bit float
    finite = np.isfinite(g) & np.isfinite(r)
    # the largest finite value and infinity are one step apart: a kernel
    # result on the other side of the overflow threshold counts as one step
    edge = ~finite & (ulp == 1) & ~np.isnan(g) & ~np.isnan(r)
    with np.errstate(invalid="ignore"):
        over_bound = (~(diff <= rel * np.abs(r) + floor) | ~finite) & ~edge
    multi_ulp = (ulp > 1) & ~((diff <= floor) & finite)
    bad = (over_bound | multi_ulp) & (gpu_bits != ref_bits)
    n = max(1, gpu_bits.size)
    unexplained = None
    if exact is not None:
        unexplained = int(((ulp == 1) & ~near_midpoint(exact, fmt)).sum())
    return {
        "one_ulp_not_at_midpoint": unexplained,
        "n": int(gpu_bits.size),
        "bad": int(bad.sum()),
        "one_ulp": int((ulp == 1).sum()),
        "one_ulp_frac": float((ulp == 1).sum()) / n,
        "near_zero_multi_ulp": int(((ulp > 1) & (diff <= floor)).sum()),
        "fmt": fmt,
        "exact": int((ulp == 0).sum()),
        "max_ulp": int(ulp.max()) if ulp.size else 0,
        "first_bad": (np.flatnonzero(bad)[:8].tolist()),
    }


def assert_parity(gpu_bits, ref_bits, what: str = "", abs_floor=None,
                  max_one_ulp_frac: float | None = None, fmt: str = "bf16", exact=None) -> dict:
    if max_one_ulp_frac is None:
        max_one_ulp_frac = MAX_ONE_ULP_FRACTION_F16 if fmt == "f16" else MAX_ONE_ULP_FRACTION
    rep = parity_report(gpu_bits, ref_bits, abs_floor, fmt, exact)
    assert rep["bad"] == 0, f"{what}: {rep['bad']} elements outside tolerance: {rep}"
    if exact is not None:
        assert rep["one_ulp_not_at_midpoint"] == 0, \
            f"{what}: one-step elements away from any rounding midpoint: {rep}"
        return rep
    assert rep["one_ulp_frac"] <= max_one_ulp_frac, \
        f"{what}: {rep['one_ulp_frac']:.5%} elements one step off (> {max_one_ulp_frac:.2%}): {rep}"
    return rep
