"""Every element of a full-size row-norm output against the oracle (tests only).

The measured workloads run to 2^29 elements a launch.  The fp64 C oracle
covers one of them in about a second when its rows are split over the host
cores (the C code releases the GIL through ctypes), so the full-size parity
tests compare every element instead of a sample of rows.  Rows are cut into
chunks of about CHUNK_ELEMS elements; each chunk runs the oracle and the
element-by-element checker of tests/parity.py on its own worker thread, and
the counts add up to the report of the whole tensor, to which the stated
bar applies: no element outside the tolerance, and at most the format's
fraction of elements one step off.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from tests.parity import MAX_ONE_ULP_FRACTION, MAX_ONE_ULP_FRACTION_F16, parity_report

CHUNK_ELEMS = 1 << 22


def host_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def assert_full_parity(got_y: np.ndarray, oracle_rows, what: str, fmt: str = "bf16",
                       got_h: np.ndarray | None = None) -> dict:
    """`got_y` (and `got_h`, the fused add's sum): the CUDA outputs as uint16
    bit patterns [M, N] on the host.  `oracle_rows(a, b)` returns the oracle's
    (h or None, y) for rows a..b-1.  h, where given, must match bit for bit."""
    M, N = got_y.shape
    step = max(1, CHUNK_ELEMS // max(1, N))
    spans = [(a, min(M, a + step)) for a in range(0, M, step)]

    def one(span):
        a, b = span
        h_want, y_want = oracle_rows(a, b)
        rep = parity_report(got_y[a:b], y_want, fmt=fmt)
        h_bad = 0
        if got_h is not None:
            h_bad = int(np.count_nonzero(got_h[a:b] != h_want))
        first = [a * N + i for i in rep["first_bad"]]
        return rep["n"], rep["bad"], rep["one_ulp"], rep["max_ulp"], h_bad, first

    with ThreadPoolExecutor(max_workers=host_threads()) as pool:
        parts = list(pool.map(one, spans))
    n = sum(p[0] for p in parts)
    bad = sum(p[1] for p in parts)
    one_ulp = sum(p[2] for p in parts)
    h_bad = sum(p[4] for p in parts)
    rep = {"n": n, "bad": bad, "one_ulp": one_ulp, "one_ulp_frac": one_ulp / max(1, n),
           "max_ulp": max((p[3] for p in parts), default=0), "h_mismatch": h_bad,
           "first_bad": [i for p in parts for i in p[5]][:8], "chunks": len(spans)}
    cap = MAX_ONE_ULP_FRACTION_F16 if fmt == "f16" else MAX_ONE_ULP_FRACTION
    assert h_bad == 0, f"{what}: {h_bad} elements of h differ from the oracle: {rep}"
    assert bad == 0, f"{what}: {bad} elements outside tolerance: {rep}"
    assert rep["one_ulp_frac"] <= cap, \
        f"{what}: {rep['one_ulp_frac']:.5%} elements one step off (> {cap:.2%}): {rep}"
    return rep
