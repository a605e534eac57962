"""The parity checker itself (CPU only): it must accept what the stated
tolerance allows and reject each kind of disagreement, in both formats."""
from __future__ import annotations

import numpy as np
import pytest

from tests.parity import parity_report


def bits(vals, fmt):
    dt = np.float16 if fmt == "f16" else np.float32
    a = np.asarray(vals, dtype=dt)
    if fmt == "f16":
        return a.view(np.uint16)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_identical_outputs_pass(fmt):
    ref = bits(np.linspace(-3, 3, 1001), fmt)
    rep = parity_report(ref, ref, fmt=fmt)
    assert rep["bad"] == 0 and rep["one_ulp"] == 0 and rep["exact"] == ref.size


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_one_step_counts_two_steps_fail(fmt):
    ref = bits(np.linspace(0.5, 3, 1000), fmt)
    one = ref.copy()
    one[::100] += 1
    rep = parity_report(one, ref, fmt=fmt)
    assert rep["bad"] == 0 and rep["one_ulp"] == 10 and rep["max_ulp"] == 1
    two = ref.copy()
    two[5] += 2
    assert parity_report(two, ref, fmt=fmt)["bad"] == 1


def test_step_sizes_differ_by_format():
    # the same value 1.0 one step up is 2^-7 away in bf16 and 2^-10 in fp16;
    # an error of 2^-9 is under one bf16 step but four fp16 steps
    ref_b, ref_h = bits([1.0], "bf16"), bits([1.0], "f16")
    assert parity_report(ref_b + 1, ref_b, fmt="bf16")["max_ulp"] == 1
    off = bits([1.0 + 2.0**-8], "f16")
    assert parity_report(off, ref_h, fmt="f16")["bad"] == 1
    # reading fp16 bits as bf16 would decode a different number: the format matters
    assert parity_report(ref_h, ref_h + 1, fmt="f16")["bad"] == 0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_near_zero_allowance_and_signed_zero(fmt):
    ref = bits([0.0, 1e-7, -0.0], fmt)
    got = bits([-0.0, -1e-7, 0.0], fmt)  # many steps apart near zero but within 1e-6
    rep = parity_report(got, ref, fmt=fmt)
    assert rep["bad"] == 0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_infinities(fmt):
    big = 65504.0 if fmt == "f16" else 3.3895313892515355e38
    ref = bits([np.inf, -np.inf, big, np.inf], fmt)
    ok = bits([np.inf, -np.inf, np.inf, big], fmt)   # equal, or across the overflow edge
    assert parity_report(ok, ref, fmt=fmt)["bad"] == 0
    wrong = bits([-np.inf, np.inf, 1.0, np.nan], fmt)
    assert parity_report(wrong, ref, fmt=fmt)["bad"] == 4
    far = bits([big / 2], fmt)
    assert parity_report(far, bits([np.inf], fmt), fmt=fmt)["bad"] == 1


def test_nan_only_matches_itself():
    ref = bits([np.nan, 1.0], "f16")
    assert parity_report(ref, ref, fmt="f16")["bad"] == 0
    assert parity_report(bits([1.0, 1.0], "f16"), ref, fmt="f16")["bad"] == 1


def test_midpoint_mode_accepts_ties_and_rejects_other_one_step_errors():
    from tests.parity import near_midpoint
    # 1 + 2^-8 is the bf16 midpoint between 1 and 1 + 2^-7
    exact = np.array([1 + 2.0**-8 + 2.0**-30, 1.25, 1 + 2.0**-8 - 2.0**-26])
    assert near_midpoint(exact).tolist() == [True, False, True]
    ref = bits([1.0 + 2.0**-7, 1.25, 1.0], "bf16")        # oracle rounding
    got = bits([1.0, 1.25 + 2.0**-7, 1.0 + 2.0**-7], "bf16")  # each one step away
    rep = parity_report(got, ref, exact=exact)
    assert rep["one_ulp_not_at_midpoint"] == 1              # only the 1.25 element
    # fp16: 1 + 2^-11 is a midpoint
    assert near_midpoint(np.array([1 + 2.0**-11]), fmt="f16").tolist() == [True]
    assert near_midpoint(np.array([1 + 2.0**-12]), fmt="f16").tolist() == [False]


def test_full_size_checker_adds_up_chunks_and_rejects_planted_errors(monkeypatch):
    # The chunked whole-tensor check (tests/full_compare.py) on an oracle
    # output: identical passes; a two-step element in a late chunk, a one-step
    # fraction above 0.1% spread over chunk boundaries, or one differing h
    # element fails, with the element's flat index reported.
    import oracle
    from tests import full_compare
    monkeypatch.setattr(full_compare, "CHUNK_ELEMS", 3 * 64)   # 3 rows a chunk
    rng = np.random.default_rng(5)
    x = bits(rng.standard_normal((40, 64)), "bf16")
    w = bits(1 + 0.1 * rng.standard_normal(64), "bf16")
    y = oracle.rmsnorm(x, w, 1e-6)
    rows = lambda a, b: (None, oracle.rmsnorm(x[a:b], w, 1e-6))  # noqa: E731
    rep = full_compare.assert_full_parity(y.copy(), rows, "same")
    assert rep["n"] == y.size and rep["bad"] == 0 and rep["chunks"] == 14
    two = y.copy()
    two[37, 5] += 2
    with pytest.raises(AssertionError, match=str(37 * 64 + 5)):
        full_compare.assert_full_parity(two, rows, "two steps")
    many = y.copy()
    many[::7, 3] += 1                                    # 6 rows of 40: 0.23% of elements
    with pytest.raises(AssertionError, match="one step off"):
        full_compare.assert_full_parity(many, rows, "fraction")
    h = x.copy()
    with pytest.raises(AssertionError, match="of h differ"):
        h_bad = h.copy()
        h_bad[20, 0] ^= 1
        full_compare.assert_full_parity(y.copy(), lambda a, b: (h[a:b], rows(a, b)[1]), "h",
                                        got_h=h_bad)
