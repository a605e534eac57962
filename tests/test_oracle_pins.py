"""Pins for the fp64 CPU oracle (CPU only).

The oracle is the yardstick for the CUDA path, so it is itself checked
against things other than itself: hand-worked rows (tests/golden), closed
forms, invariants, exact rational arithmetic on tiny inputs, and a numpy
restatement.  Each pin is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, eps in the wrong place, a double
rounding) fails at least one of them.

Operations: RMSNorm ("[Inductor] Codegen Gluon", section 3.1); fused Q/K
RMSNorm + neox RoPE ("[pretuned] Optimize fused_qk_norm_rope on B200",
section "Summary"); LayerNorm ("TorchInductor: from ATen IR to Triton
kernel", section 14.12.2).
"""
from __future__ import annotations

import math
import os
import struct
from decimal import Decimal
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.exact import (bits_to_f64, bits_to_fraction, dcos, dec_to_f32, dsin,
                         dsqrt, f32_to_fraction, round_bf16, to_dec)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(vals) -> np.ndarray:
    """Python floats exactly representable in bf16 -> bit patterns."""
    out = []
    for v in vals:
        u = struct.unpack("<I", struct.pack("<f", float(v)))[0]
        assert u & 0xFFFF == 0, f"{v} is not a bf16 value"
        out.append(u >> 16)
    return np.array(out, dtype=np.uint16)


def rand_bf16(rng, shape, scale=1.0) -> np.ndarray:
    x = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_of(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

class TestBf16Rounding:
    def test_ties_go_to_even(self):
        # 1 + 2^-8 lies halfway between 1 (even) and 1 + 2^-7 (odd): -> 1
        assert oracle.double_to_bf16(1 + 2**-8) == 0x3F80
        # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
        assert oracle.double_to_bf16(1 + 3 * 2**-8) == 0x3F82
        assert oracle.double_to_bf16(-(1 + 2**-8)) == 0xBF80

    def test_single_rounding_not_via_float(self):
        # Just above the tie: direct rounding goes up.  Rounding to binary32
        # first would land exactly on the tie and then go down to 1.0.
        assert oracle.double_to_bf16(1 + 2**-8 + 2**-40) == 0x3F81
        assert oracle.double_to_bf16(1 + 2**-8 - 2**-40) == 0x3F80

    def test_matches_library_on_binary32_values(self):
        # A binary32 value rounds to bf16 in one step both ways, so the oracle
        # must agree with torch's float32 -> bfloat16 conversion (RNE).
        rng = np.random.default_rng(7)
        u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
        f = u.view(np.float32)
        f = f[np.isfinite(f)]
        lib = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ours = np.array([oracle.double_to_bf16(float(v)) for v in f], dtype=np.uint16)
        # torch keeps NaN payloads / may round huge values to inf the same way
        assert np.array_equal(ours, lib)

    def test_subnormals_and_overflow(self):
        assert oracle.double_to_bf16(2.0**-133) == 0x0001
        assert oracle.double_to_bf16(2.0**-134) == 0x0000      # tie -> even (0)
        assert oracle.double_to_bf16(1.5 * 2.0**-133) == 0x0002  # tie -> even (2)
        assert oracle.double_to_bf16(3.39e38) == 0x7F7F        # largest finite
        assert oracle.double_to_bf16(2.0**128 - 2.0**119) == 0x7F80  # tie -> inf
        assert oracle.double_to_bf16(-1e39) == 0xFF80
        assert oracle.double_to_bf16(-0.0) == 0x8000

    def test_matches_exact_rational_rounding(self):
        rng = np.random.default_rng(11)
        vals = rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000))
        for v in vals:
            assert oracle.double_to_bf16(float(v)) == round_bf16(Fraction(float(v)))


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def _parse_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([f.strip() for f in line.split("|")])
    return rows


@pytest.mark.parametrize("row", _parse_golden("rmsnorm_hand.txt"), ids=lambda r: r[0])
def test_rmsnorm_hand_worked(row):
    _, eps, xs, ws, ys = row
    x = bf([float(v) for v in xs.split()])[None, :]
    w = bf([float(v) for v in ws.split()])
    want = np.array([int(h, 16) for h in ys.split()], dtype=np.uint16)
    got = oracle.rmsnorm(x, w, float(eps))[0]
    assert [hex(v) for v in got] == [hex(v) for v in want]


@pytest.mark.parametrize("c", [1.0, -3.5, 0.0009994507, 96.0])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5])
def test_rmsnorm_constant_row_closed_form(c, eps):
    # Constant row c: mean(x^2) = c^2, so y_j = sign(c) * w_j * |c| / sqrt(c^2 + eps).
    # The 0.0009994507 row (c^2 ~ 1e-6) is where eps placement matters.
    N = 37
    rng = np.random.default_rng(3)
    cb = bf([c])[0]
    cq = bits_to_fraction(cb)
    x = np.full((1, N), cb, dtype=np.uint16)
    w = rand_bf16(rng, (N,))
    got = oracle.rmsnorm(x, w, eps)[0]
    epsq = f32_to_fraction(eps)
    denom = dsqrt(cq * cq + epsq)
    for j in range(N):
        wq = bits_to_fraction(w[j])
        want = round_bf16(to_dec(wq * cq) / denom)
        assert got[j] == want, (j, hex(got[j]), hex(want))


def test_rmsnorm_one_hot_closed_form():
    N = 64
    rng = np.random.default_rng(5)
    w = rand_bf16(rng, (N,))
    for k, a in [(0, 5.0), (17, -0.125), (63, 300.0)]:
        x = np.zeros((1, N), dtype=np.uint16)
        x[0, k] = bf([a])[0]
        eps = 1e-6
        got = oracle.rmsnorm(x, w, eps)[0]
        aq = Fraction(a)
        want_k = round_bf16(to_dec(bits_to_fraction(w[k]) * aq) /
                            dsqrt(aq * aq / N + f32_to_fraction(eps)))
        assert got[k] == want_k
        others = np.delete(bits_to_f64(got), k)
        assert np.all(others == 0.0)


def test_rmsnorm_unit_rms_invariant():
    # With eps = 0, sum_j (x_j * rstd)^2 = N exactly in real arithmetic; the
    # per-row statistic must give that to double precision, and the bf16
    # outputs (w = 1) must give it to within bf16 rounding.
    rng = np.random.default_rng(9)
    x = rand_bf16(rng, (6, 300), scale=4.0)
    rstd = oracle.rms_rstd(x, 0.0)
    xf = bits_to_f64(x)
    s = ((xf * rstd[:, None]) ** 2).sum(axis=1)
    np.testing.assert_allclose(s, 300.0, rtol=1e-12)
    w = bf([1.0] * 300)
    y = bits_to_f64(oracle.rmsnorm(x, w, 0.0))
    np.testing.assert_allclose((y * y).sum(axis=1), 300.0, rtol=2**-7)


@pytest.mark.parametrize("eps", [1e-6, 1e-5, 0.25])
def test_rms_rstd_against_exact_decimal(eps):
    # The row statistic alone, with eps > 0: rstd = 1/sqrt(sum(x^2)/N + eps)
    # against 60-digit decimals on exact rationals (x and eps as the binary
    # values the oracle receives).  Rows of three scales, including values
    # near 1e-3 where x^2 ~ eps and eps's placement (inside the root, on the
    # mean, not on the sum) moves rstd by far more than double rounding.
    rng = np.random.default_rng(31)
    epsq = f32_to_fraction(eps)
    for N, scale in [(1, 1.0), (7, 1e-3), (64, 1e-3), (300, 1.0), (129, 30.0)]:
        x = rand_bf16(rng, (3, N), scale=scale)
        got = oracle.rms_rstd(x, eps)
        for r in range(3):
            ms = sum(bits_to_fraction(v) ** 2 for v in x[r]) / N
            want = Decimal(1) / dsqrt(ms + epsq)
            assert abs(Decimal(float(got[r])) - want) <= want * Decimal("1e-14"), (N, r)
    # constant row c: rstd = 1/sqrt(c^2 + eps) whatever N is
    cb = bf([0.0009994507])[0]
    cq = bits_to_fraction(cb)
    for N in (1, 5, 4096):
        got = oracle.rms_rstd(np.full((1, N), cb, dtype=np.uint16), eps)[0]
        want = Decimal(1) / dsqrt(cq * cq + epsq)
        assert abs(Decimal(float(got)) - want) <= want * Decimal("1e-14"), N


def test_rmsnorm_power_of_two_scale_is_exact():
    # eps = 0: scaling a row by 2^k scales mean(x^2) by 4^k and rstd by 2^-k,
    # all exact in binary arithmetic, so the outputs are bit-identical.
    rng = np.random.default_rng(13)
    x = rand_bf16(rng, (4, 256))
    w = rand_bf16(rng, (256,))
    y0 = oracle.rmsnorm(x, w, 0.0)
    for k in (-20, -3, 5, 40):
        xs = (x.astype(np.int32) + (k << 7)).astype(np.uint16)  # add k to the exponent
        assert np.array_equal(bits_to_f64(xs), bits_to_f64(x) * 2.0**k)
        assert np.array_equal(oracle.rmsnorm(xs, w, 0.0), y0)


def test_rmsnorm_outlier_scale_nearly_invariant():
    # The outlier rows of the sweep are x * 100: with eps = 1e-6 the result may
    # move by at most one bf16 step.
    rng = np.random.default_rng(17)
    xf = rng.standard_normal((8, 512)).astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    x100 = (torch.from_numpy(xf) * 100).to(torch.bfloat16)
    to_bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    w = rand_bf16(rng, (512,))
    y = bits_to_f64(oracle.rmsnorm(to_bits(x), w, 1e-6))
    y100 = bits_to_f64(oracle.rmsnorm(to_bits(x100), w, 1e-6))
    # inputs themselves differ by a bf16 rounding, so allow 2^-6 relative
    np.testing.assert_allclose(y100, y, rtol=2**-6, atol=1e-30)


def test_rmsnorm_exact_brute_force():
    rng = np.random.default_rng(21)
    for N in (1, 2, 3, 5, 8, 13, 16):
        for eps in (0.0, 1e-6, 0.5):
            x = rand_bf16(rng, (3, N), scale=2.0)
            w = rand_bf16(rng, (N,))
            got = oracle.rmsnorm(x, w, eps)
            epsq = f32_to_fraction(eps)
            for r in range(3):
                xs = [bits_to_fraction(v) for v in x[r]]
                ms = sum(v * v for v in xs) / N
                if ms + epsq == 0:
                    continue
                den = dsqrt(ms + epsq)
                for j in range(N):
                    want = round_bf16(to_dec(xs[j] * bits_to_fraction(w[j])) / den)
                    assert got[r, j] == want, (N, eps, r, j)


def test_rmsnorm_matches_numpy_restatement():
    rng = np.random.default_rng(23)
    x = rand_bf16(rng, (8, 520))
    w = rand_bf16(rng, (520,))
    eps = 1e-6
    xf = bits_to_f64(x)
    wf = bits_to_f64(w)
    ref = xf * (1.0 / np.sqrt((xf * xf).mean(-1, keepdims=True) + np.float64(np.float32(eps)))) * wf
    want = np.array([[round_bf16(Fraction(float(v))) for v in row] for row in ref], dtype=np.uint16)
    got = oracle.rmsnorm(x, w, eps)
    assert np.array_equal(got, want)


def test_rmsnorm_rejects_bad_shapes():
    with pytest.raises(oracle.OracleError):
        oracle.rmsnorm(np.zeros((2, 0), np.uint16), np.zeros(0, np.uint16), 1e-6)
    assert oracle.rmsnorm(np.zeros((0, 8), np.uint16), np.zeros(8, np.uint16), 1e-6).shape == (0, 8)


# ---------------------------------------------------------------------------
# rotary table
# ---------------------------------------------------------------------------

class TestRopeTable:
    def test_position_zero_is_identity(self):
        t = oracle.rope_cos_sin(1e6, 4, 128)
        assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)

    def test_unit_circle(self):
        t = oracle.rope_cos_sin(1e6, 2048, 64).astype(np.float64)
        c, s = t[:, :32], t[:, 32:]
        assert np.max(np.abs(c * c + s * s - 1.0)) < 2**-22

    @pytest.mark.parametrize("theta,r,p,i", [(10000.0, 4, 1, 0), (10000.0, 4, 1, 1),
                                             (1e6, 128, 131071, 0), (1e6, 128, 131071, 5),
                                             (1e6, 64, 99991, 31), (1e6, 128, 7, 63)])
    def test_entries_against_decimal(self, theta, r, p, i):
        # cos/sin of p * theta^(-2i/r), evaluated with 60-digit decimals and
        # rounded to binary32.  Also pins the frequency exponent (-2i/r, r not D).
        t = oracle.rope_cos_sin(theta, p + 1, r)
        f = Decimal(theta) ** (Decimal(-2 * i) / Decimal(r))
        a = Decimal(p) * f
        assert t[p, i] == np.float32(dec_to_f32(dcos(a)))
        assert t[p, r // 2 + i] == np.float32(dec_to_f32(dsin(a)))

    def test_hand_values(self):
        # theta = 10000, r = 4: f_0 = 1, f_1 = 10000^(-1/2) = 0.01
        t = oracle.rope_cos_sin(10000.0, 3, 4)
        assert abs(t[1, 0] - math.cos(1.0)) < 1e-7
        assert abs(t[1, 1] - math.cos(0.01)) < 1e-7
        assert abs(t[2, 3] - math.sin(0.02)) < 1e-7

    # The bf16 table: the same angles, each entry rounded once to bf16.

    def test_bf16_position_zero_is_identity(self):
        t = oracle.rope_cos_sin_bf16(1e6, 4, 128)
        assert np.all(t[0, :64] == 0x3F80) and np.all(t[0, 64:] == 0)

    def test_bf16_unit_circle(self):
        t = bits_to_f64(oracle.rope_cos_sin_bf16(1e6, 2048, 64))
        c, s = t[:, :32], t[:, 32:]
        # each entry within half a bf16 step (2^-9 relative): c^2 + s^2 within 2^-7 of 1
        assert np.max(np.abs(c * c + s * s - 1.0)) < 2**-7

    @pytest.mark.parametrize("theta,r,p,i", [(10000.0, 4, 1, 0), (10000.0, 4, 1, 1),
                                             (1e6, 128, 131071, 0), (1e6, 128, 131071, 5),
                                             (1e6, 64, 99991, 31), (1e6, 128, 7, 63)])
    def test_bf16_entries_against_decimal(self, theta, r, p, i):
        t = oracle.rope_cos_sin_bf16(theta, p + 1, r)
        a = Decimal(p) * Decimal(theta) ** (Decimal(-2 * i) / Decimal(r))
        assert t[p, i] == round_bf16(dcos(a))
        assert t[p, r // 2 + i] == round_bf16(dsin(a))

    @pytest.mark.parametrize("p,col", [(137, 59), (1247, 50), (6883, 60), (6985, 16)])
    def test_bf16_entries_rounded_once(self, p, col):
        # At these entries (theta 1e6, r 64) the binary32 value lies exactly
        # halfway between two bf16 values and ties to the even one, which is
        # not the bf16 nearest the exact value: a table rounded through
        # binary32 would differ here.
        r, half = 64, 32
        k = col % half
        a = Decimal(p) * Decimal(1e6) ** (Decimal(-2 * k) / Decimal(r))
        exact = dcos(a) if col < half else dsin(a)
        t = oracle.rope_cos_sin_bf16(1e6, p + 1, r)
        assert t[p, col] == round_bf16(exact)
        f32 = int(oracle.rope_cos_sin(1e6, p + 1, r).view(np.uint32)[p, col])
        assert f32 & 0xFFFF == 0x8000
        twice = (f32 >> 16) + ((f32 >> 16) & 1)  # ties to even from the binary32 value
        assert twice != t[p, col]


# ---------------------------------------------------------------------------
# fused Q/K RMSNorm + neox RoPE
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("row", _parse_golden("qk_norm_rope_hand.txt"), ids=lambda r: r[0])
def test_qk_hand_worked(row):
    _, eps, D, r, xs, ws, cs, want = row
    D, r = int(D), int(r)
    x = bf([float(v) for v in xs.split()])
    w = bf([float(v) for v in ws.split()])
    table = np.array([[float(v) for v in cs.split()]], dtype=np.float32)
    want = np.array([int(h, 16) for h in want.split()], dtype=np.uint16)
    # one token, one query head, no key heads
    qkv = x[None, :]
    got = oracle.qk_norm_rope(qkv, w, w, table, np.array([0]), 1, 0, D, r, float(eps))
    assert [hex(v) for v in got[0]] == [hex(v) for v in want]


def _norm_only(head_bits, w, eps):
    return oracle.rmsnorm(head_bits[None, :], w, eps)[0]


def _layout(T, Hq, Hkv, D, rng):
    qkv = rand_bf16(rng, (T, (Hq + 2 * Hkv) * D))
    wq = rand_bf16(rng, (D,))
    wk = rand_bf16(rng, (D,))
    return qkv, wq, wk


def test_qk_position_zero_is_norm_only_and_v_untouched():
    rng = np.random.default_rng(31)
    T, Hq, Hkv, D, r = 3, 4, 2, 16, 16
    qkv, wq, wk = _layout(T, Hq, Hkv, D, rng)
    table = oracle.rope_cos_sin(1e6, 8, r)
    out = oracle.qk_norm_rope(qkv, wq, wk, table, np.zeros(T, np.int64), Hq, Hkv, D, r, 1e-6)
    for t in range(T):
        for h in range(Hq + 2 * Hkv):
            src = qkv[t, h * D:(h + 1) * D]
            dst = out[t, h * D:(h + 1) * D]
            if h < Hq:
                assert np.array_equal(dst, _norm_only(src, wq, 1e-6))
            elif h < Hq + Hkv:
                assert np.array_equal(dst, _norm_only(src, wk, 1e-6))
            else:
                assert np.array_equal(dst, src)  # value head: bit-identical


def _flip(bits):
    return (bits ^ 0x8000).astype(np.uint16)


@pytest.mark.parametrize("D,r", [(16, 16), (16, 8), (8, 4), (128, 64), (128, 128)])
def test_qk_quarter_turn_permutes_pairs(D, r):
    # cos = 0, sin = 1: o_i = -n_{i+r/2}, o_{i+r/2} = n_i, tail unchanged.  Pins
    # the partner index (i + r/2, not i + D/2), both signs and the tail.
    rng = np.random.default_rng(37)
    Hq, Hkv = 2, 1
    qkv, wq, wk = _layout(1, Hq, Hkv, D, rng)
    h2 = r // 2
    table = np.concatenate([np.zeros(h2), np.ones(h2)]).astype(np.float32)[None, :]
    out = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([0]), Hq, Hkv, D, r, 1e-6)
    for h in range(Hq + Hkv):
        n = _norm_only(qkv[0, h * D:(h + 1) * D], wq if h < Hq else wk, 1e-6)
        o = out[0, h * D:(h + 1) * D]
        assert np.array_equal(o[:h2], _flip(n[h2:r]))
        assert np.array_equal(o[h2:r], n[:h2])
        assert np.array_equal(o[r:], n[r:])


def test_qk_query_and_key_weights_are_separate():
    rng = np.random.default_rng(41)
    D = 32
    x = rand_bf16(rng, (D,))
    qkv = np.concatenate([x, x, x])[None, :]  # Hq=1, Hkv=1: q, k, v identical
    wq = bf([1.0] * D)
    wk = bf([2.0] * D)
    table = oracle.rope_cos_sin(1e6, 4, D)
    out = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([3]), 1, 1, D, D, 1e-6)
    q, k, v = out[0, :D], out[0, D:2 * D], out[0, 2 * D:]
    assert np.array_equal(bits_to_f64(k), 2.0 * bits_to_f64(q))
    assert np.array_equal(v, x)


def test_qk_exact_brute_force():
    # Exact rationals for the table and inputs, 60-digit decimals for rstd;
    # the oracle must round to the same bf16 for every element.
    rng = np.random.default_rng(43)
    for D, r in [(8, 8), (8, 4), (8, 2), (6, 4)]:
        Hq, Hkv, T = 2, 1, 2
        qkv, wq, wk = _layout(T, Hq, Hkv, D, rng)
        maxp = 5
        table = rng.standard_normal((maxp, r)).astype(np.float32)  # any numbers work
        pos = np.array([4, 1], dtype=np.int64)
        eps = 1e-6
        out = oracle.qk_norm_rope(qkv, wq, wk, table, pos, Hq, Hkv, D, r, eps)
        h2 = r // 2
        for t in range(T):
            cs = [Fraction(float(v)) for v in table[pos[t]]]
            for h in range(Hq + Hkv):
                w = wq if h < Hq else wk
                xs = [bits_to_fraction(v) for v in qkv[t, h * D:(h + 1) * D]]
                ws = [bits_to_fraction(v) for v in w]
                den = dsqrt(sum(v * v for v in xs) / D + f32_to_fraction(eps))
                # n_j = x_j w_j / den: keep the rational numerator, divide once
                a = [xs[j] * ws[j] for j in range(D)]
                o = list(a)
                for i in range(h2):
                    o[i] = a[i] * cs[i] - a[i + h2] * cs[h2 + i]
                    o[i + h2] = a[i + h2] * cs[i] + a[i] * cs[h2 + i]
                want = [round_bf16(to_dec(v) / den) for v in o]
                got = list(out[t, h * D:(h + 1) * D])
                assert got == want, (D, r, t, h)


def test_qk_rotation_preserves_pair_norm():
    rng = np.random.default_rng(47)
    D, r = 128, 128
    qkv, wq, wk = _layout(4, 4, 2, D, rng)
    table = oracle.rope_cos_sin(1e6, 1000, r)
    pos = np.array([0, 17, 500, 999], dtype=np.int64)
    out = oracle.qk_norm_rope(qkv, wq, wk, table, pos, 4, 2, D, r, 1e-6)
    h2 = r // 2
    for t in range(4):
        for h in range(6):
            n = bits_to_f64(_norm_only(qkv[t, h * D:(h + 1) * D], wq if h < 4 else wk, 1e-6))
            o = bits_to_f64(out[t, h * D:(h + 1) * D])
            pn = n[:h2] ** 2 + n[h2:r] ** 2
            po = o[:h2] ** 2 + o[h2:r] ** 2
            # each side carries up to 2^-8 relative rounding per element
            assert np.all(np.abs(po - pn) <= 2**-6 * pn + 1e-12)


def test_qk_relative_position_dot_product():
    # <R_p q, R_s k> depends only on p - s.  Compare (p, s) with (p+d, s+d).
    rng = np.random.default_rng(53)
    D = r = 64
    x = rand_bf16(rng, (2 * D,))
    qkv = np.concatenate([x, rand_bf16(rng, (D,))])[None, :]  # q, k, v of one token
    wq = wk = bf([1.0] * D)
    table = oracle.rope_cos_sin(10000.0, 4096, r)

    def dot(p, s):
        a = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([p]), 1, 1, D, r, 1e-6)
        b = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([s]), 1, 1, D, r, 1e-6)
        return float(np.dot(bits_to_f64(a[0, :D]), bits_to_f64(b[0, D:2 * D])))

    for p, s, d in [(5, 2, 100), (300, 1000, 2000), (0, 0, 3000)]:
        d0, d1 = dot(p, s), dot(p + d, s + d)
        # q, k unit-RMS (norm ~ 8): the dot products agree to bf16 accuracy
        assert abs(d0 - d1) <= 0.05 * D ** 0.5 + 2**-6 * abs(d0)
    # and the dot product does change with p - s (the test is not vacuous)
    assert abs(dot(5, 2) - dot(50, 2)) > 0.1


def test_qk_rejects_out_of_range_position():
    rng = np.random.default_rng(59)
    qkv, wq, wk = _layout(2, 1, 1, 8, rng)
    table = oracle.rope_cos_sin(1e6, 4, 8)
    with pytest.raises(oracle.OracleError):
        oracle.qk_norm_rope(qkv, wq, wk, table, np.array([0, 4]), 1, 1, 8, 8, 1e-6)
    with pytest.raises(oracle.OracleError):
        oracle.qk_norm_rope(qkv, wq, wk, table, np.array([-1, 0]), 1, 1, 8, 8, 1e-6)


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

def test_layernorm_constant_row_gives_bias():
    N = 24
    rng = np.random.default_rng(61)
    w = rand_bf16(rng, (N,))
    b = rand_bf16(rng, (N,))
    x = np.full((2, N), bf([3.25])[0], dtype=np.uint16)
    y = oracle.layernorm(x, w, b, 1e-5)
    assert np.array_equal(y[0], b) and np.array_equal(y[1], b)


def test_layernorm_two_point_closed_form():
    # row [a, -a, a, -a]: mean 0, var a^2, y = +-a/sqrt(a^2+eps) * w + b
    a = 1.5
    x = bf([a, -a, a, -a])[None, :]
    w = bf([1.0, 2.0, 0.5, 1.0])
    b = bf([0.0, 0.0, 0.0, 1.0])
    eps = 1e-5
    y = oracle.layernorm(x, w, b, eps)[0]
    den = dsqrt(Fraction(a) ** 2 + f32_to_fraction(eps))
    for j, sgn in enumerate([1, -1, 1, -1]):
        want = round_bf16(to_dec(sgn * Fraction(a) * bits_to_fraction(w[j])) / den
                          + to_dec(bits_to_fraction(b[j])))
        assert y[j] == want


def test_layernorm_exact_brute_force_and_numpy():
    rng = np.random.default_rng(67)
    for N in (2, 3, 7, 16):
        x = rand_bf16(rng, (3, N), scale=3.0)
        x = (x.astype(np.int32)).astype(np.uint16)
        w = rand_bf16(rng, (N,))
        b = rand_bf16(rng, (N,))
        eps = 1e-5
        got = oracle.layernorm(x, w, b, eps)
        for r in range(3):
            xs = [bits_to_fraction(v) for v in x[r]]
            mean = sum(xs) / N
            var = sum((v - mean) ** 2 for v in xs) / N
            den = dsqrt(var + f32_to_fraction(eps))
            for j in range(N):
                want = round_bf16(to_dec((xs[j] - mean) * bits_to_fraction(w[j])) / den
                                  + to_dec(bits_to_fraction(b[j])))
                assert got[r, j] == want
    # numpy restatement (np.var is the biased variance)
    x = rand_bf16(rng, (4, 300))
    w = rand_bf16(rng, (300,))
    xf = bits_to_f64(x)
    ref = (xf - xf.mean(-1, keepdims=True)) / np.sqrt(xf.var(-1, keepdims=True) + np.float64(np.float32(1e-5))) * bits_to_f64(w)
    want = np.array([[round_bf16(Fraction(float(v))) for v in row] for row in ref], dtype=np.uint16)
    got = oracle.layernorm(x, w, None, 1e-5)
    mism = np.count_nonzero(got != want)
    assert mism == 0


# ---------------------------------------------------------------------------
# fused residual add + RMSNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("row", _parse_golden("add_rmsnorm_hand.txt"), ids=lambda r: r[0])
def test_add_rmsnorm_hand_worked(row):
    _, eps, xs, rs, ws, hs, ys = row
    x = bf([float(v) for v in xs.split()])[None, :]
    r = bf([float(v) for v in rs.split()])[None, :]
    w = bf([float(v) for v in ws.split()])
    h, y = oracle.add_rmsnorm(x, r, w, float(eps))
    assert [hex(v) for v in h[0]] == [hex(int(t, 16)) for t in hs.split()]
    assert [hex(v) for v in y[0]] == [hex(int(t, 16)) for t in ys.split()]


def test_add_rmsnorm_sum_is_the_correctly_rounded_sum():
    # h must be the single rounding of the exact sum: compare with exact
    # rationals, and with torch's bf16 addition (library routine).
    rng = np.random.default_rng(71)
    x = rand_bf16(rng, (16, 64), scale=3.0)
    r = rand_bf16(rng, (16, 64), scale=0.01)
    r[:, :8] = (x[:, :8] ^ 0x8000)               # exact cancellation
    r[:, 8:16] = rand_bf16(rng, (16, 8), scale=1e-6)  # far smaller addend
    w = rand_bf16(rng, (64,))
    h, _ = oracle.add_rmsnorm(x, r, w, 1e-6)
    for i in range(16):
        for j in range(64):
            assert h[i, j] == round_bf16(bits_to_fraction(x[i, j]) + bits_to_fraction(r[i, j]))
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    tr = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16)
    th = (tx + tr).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(np.where(bits_to_f64(h) == 0, 0, h), np.where(bits_to_f64(th) == 0, 0, th))


def test_add_rmsnorm_is_the_composition():
    # The fused op changes nothing: y equals RMSNorm of the rounded sum, bit for
    # bit, on random rows (which also catches a y taken from the unrounded sum).
    rng = np.random.default_rng(73)
    x = rand_bf16(rng, (32, 257 * 8))
    r = rand_bf16(rng, (32, 257 * 8), scale=0.5)
    w = rand_bf16(rng, (257 * 8,))
    h, y = oracle.add_rmsnorm(x, r, w, 1e-6)
    assert np.array_equal(y, oracle.rmsnorm(h, w, 1e-6))
    # and y is NOT what the unrounded sum would give on at least some elements
    xf, rf, wf = bits_to_f64(x), bits_to_f64(r), bits_to_f64(w)
    s = xf + rf
    unrounded = s / np.sqrt((s * s).mean(-1, keepdims=True) + np.float64(np.float32(1e-6))) * wf
    yu = np.array([[round_bf16(Fraction(float(v))) for v in row] for row in unrounded[:4]],
                  dtype=np.uint16)
    assert np.count_nonzero(yu != y[:4]) > 0


# ---------------------------------------------------------------------------
# L2Norm
# ---------------------------------------------------------------------------

def test_l2norm_closed_forms():
    N = 64
    eps = 1e-12
    # constant row c: ||x|| = |c| sqrt(N) -> y = sign(c) / 8 exactly
    for c in (3.0, -0.5):
        y = oracle.l2norm(np.full((1, N), bf([c])[0], dtype=np.uint16), eps)[0]
        assert np.all(bits_to_f64(y) == np.sign(c) / 8.0)
    # one-hot: y = sign(a) at k, zero elsewhere
    x = np.zeros((1, N), dtype=np.uint16)
    x[0, 5] = bf([-7.25])[0]
    y = bits_to_f64(oracle.l2norm(x, eps)[0])
    assert y[5] == -1.0 and np.all(np.delete(y, 5) == 0.0)
    # a row whose norm is below eps is divided by eps, not by its norm
    x = np.full((1, 4), bf([2.0**-20])[0], dtype=np.uint16)  # ||x|| = 2^-19
    y = bits_to_f64(oracle.l2norm(x, 2.0**-10)[0])
    assert np.all(y == 2.0**-10)
    # norm = eps / 2: max(norm, eps) = eps gives 0.25; adding eps would give 1/6
    x = np.full((1, 4), bf([2.0**-11])[0], dtype=np.uint16)  # ||x|| = 2^-10
    y = bits_to_f64(oracle.l2norm(x, 2.0**-9)[0])
    assert np.all(y == 0.25)
    # zero row stays zero
    assert np.all(oracle.l2norm(np.zeros((2, 8), np.uint16), eps) == 0)


def test_l2norm_unit_norm_and_exact_brute_force():
    rng = np.random.default_rng(81)
    x = rand_bf16(rng, (5, 300), scale=2.0)
    y = bits_to_f64(oracle.l2norm(x, 1e-12))
    np.testing.assert_allclose((y * y).sum(-1), 1.0, rtol=2**-7)
    for N in (1, 3, 8, 13):
        x = rand_bf16(rng, (2, N))
        got = oracle.l2norm(x, 1e-12)
        for r in range(2):
            xs = [bits_to_fraction(v) for v in x[r]]
            den = dsqrt(sum(v * v for v in xs))
            for j in range(N):
                assert got[r, j] == round_bf16(to_dec(xs[j]) / den)


def test_l2norm_matches_library_normalize():
    # torch.nn.functional.normalize in float64 (a library routine), rounded once
    rng = np.random.default_rng(83)
    x = rand_bf16(rng, (6, 520))
    xf = torch.from_numpy(bits_to_f64(x))
    ref = torch.nn.functional.normalize(xf, p=2.0, dim=-1, eps=1e-12).numpy()
    want = np.array([[round_bf16(Fraction(float(v))) for v in row] for row in ref], dtype=np.uint16)
    assert np.array_equal(oracle.l2norm(x, 1e-12), want)


# ---------------------------------------------------------------------------
# GPT-J (interleaved) rotary pairing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D,r", [(16, 16), (16, 8), (128, 64)])
def test_gptj_quarter_turn_swaps_neighbours(D, r):
    # cos = 0, sin = 1: o_{2i} = -n_{2i+1}, o_{2i+1} = n_{2i}; the tail passes
    rng = np.random.default_rng(91)
    qkv, wq, wk = _layout(1, 2, 1, D, rng)
    h2 = r // 2
    table = np.concatenate([np.zeros(h2), np.ones(h2)]).astype(np.float32)[None, :]
    out = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([0]), 2, 1, D, r, 1e-6, style=1)
    for h in range(3):
        n = _norm_only(qkv[0, h * D:(h + 1) * D], wq if h < 2 else wk, 1e-6)
        o = out[0, h * D:(h + 1) * D]
        assert np.array_equal(o[0:r:2], _flip(n[1:r:2]))
        assert np.array_equal(o[1:r:2], n[0:r:2])
        assert np.array_equal(o[r:], n[r:])


def test_gptj_exact_brute_force_and_position_zero():
    rng = np.random.default_rng(93)
    for D, r in [(8, 8), (8, 4), (6, 2)]:
        qkv, wq, wk = _layout(2, 2, 1, D, rng)
        table = rng.standard_normal((5, r)).astype(np.float32)
        pos = np.array([3, 0], dtype=np.int64)
        out = oracle.qk_norm_rope(qkv, wq, wk, table, pos, 2, 1, D, r, 1e-6, style=1)
        h2 = r // 2
        for t in range(2):
            cs = [Fraction(float(v)) for v in table[pos[t]]]
            for h in range(3):
                w = wq if h < 2 else wk
                xs = [bits_to_fraction(v) for v in qkv[t, h * D:(h + 1) * D]]
                den = dsqrt(sum(v * v for v in xs) / D + f32_to_fraction(1e-6))
                a = [xs[j] * bits_to_fraction(w[j]) for j in range(D)]
                o = list(a)
                for i in range(h2):
                    o[2 * i] = a[2 * i] * cs[i] - a[2 * i + 1] * cs[h2 + i]
                    o[2 * i + 1] = a[2 * i + 1] * cs[i] + a[2 * i] * cs[h2 + i]
                want = [round_bf16(to_dec(v) / den) for v in o]
                assert list(out[t, h * D:(h + 1) * D]) == want
    # identity row: GPT-J and neox agree at position 0
    qkv, wq, wk = _layout(1, 2, 1, 16, rng)
    table = oracle.rope_cos_sin(1e6, 4, 16)
    a = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([0]), 2, 1, 16, 16, 1e-6, style=1)
    b = oracle.qk_norm_rope(qkv, wq, wk, table, np.array([0]), 2, 1, 16, 16, 1e-6, style=0)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# IEEE fp16 element format
# ---------------------------------------------------------------------------

from tests.exact import f16_bits_to_f64, round_f16  # noqa: E402


class TestF16Rounding:
    def test_edges(self):
        assert oracle.double_to_f16(1 + 2**-11) == 0x3C00          # tie -> even
        assert oracle.double_to_f16(1 + 3 * 2**-11) == 0x3C02      # tie -> even
        assert oracle.double_to_f16(1 + 2**-11 + 2**-40) == 0x3C01  # single rounding
        assert oracle.double_to_f16(2.0**-24) == 0x0001            # smallest subnormal
        assert oracle.double_to_f16(2.0**-25) == 0x0000            # tie -> even (0)
        assert oracle.double_to_f16(1.5 * 2.0**-24) == 0x0002      # tie -> even (2)
        assert oracle.double_to_f16(2.0**-14) == 0x0400            # smallest normal
        assert oracle.double_to_f16(65504.0) == 0x7BFF
        assert oracle.double_to_f16(65519.99) == 0x7BFF
        assert oracle.double_to_f16(65520.0) == 0x7C00             # tie -> 2^16 -> inf
        assert oracle.double_to_f16(-1e9) == 0xFC00
        assert oracle.double_to_f16(-0.0) == 0x8000

    def test_decode_every_pattern_matches_numpy(self):
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        ref = bits.view(np.float16).astype(np.float64)
        ours = np.array([oracle.f16_to_double(int(b)) for b in bits])
        same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
        assert same.all()

    def test_binary32_values_match_torch(self):
        rng = np.random.default_rng(101)
        f = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))).astype(np.float32)
        lib = torch.from_numpy(f).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
        ours = np.array([oracle.double_to_f16(float(v)) for v in f], dtype=np.uint16)
        assert np.array_equal(ours, lib)

    def test_doubles_match_exact_rationals(self):
        rng = np.random.default_rng(103)
        vals = rng.standard_normal(3000) * np.exp(rng.uniform(-18, 11, 3000))
        for v in vals:
            assert oracle.double_to_f16(float(v)) == round_f16(Fraction(float(v)))


def rand_f16(rng, shape, scale=1.0) -> np.ndarray:
    return (rng.standard_normal(shape) * scale).astype(np.float16).view(np.uint16)


def test_f16_row_ops_exact_brute_force():
    rng = np.random.default_rng(107)
    for N in (1, 3, 8, 13):
        x = rand_f16(rng, (2, N), 2.0)
        r = rand_f16(rng, (2, N), 0.5)
        w = rand_f16(rng, (N,))
        b = rand_f16(rng, (N,), 0.1)
        eps = 1e-6
        y = oracle.rmsnorm(x, w, eps, f16=True)
        h, ya = oracle.add_rmsnorm(x, r, w, eps, f16=True)
        yl = oracle.layernorm(x, w, b, eps, f16=True)
        y2 = oracle.l2norm(x, 1e-12, f16=True)
        for i in range(2):
            xs = [Fraction(float(v)) for v in x[i].view(np.float16)]
            ws = [Fraction(float(v)) for v in w.view(np.float16)]
            bs = [Fraction(float(v)) for v in b.view(np.float16)]
            den = dsqrt(sum(v * v for v in xs) / N + f32_to_fraction(eps))
            assert list(y[i]) == [round_f16(to_dec(xs[j] * ws[j]) / den) for j in range(N)]
            hs = [round_f16(xs[j] + Fraction(float(r[i].view(np.float16)[j]))) for j in range(N)]
            assert list(h[i]) == hs
            mean = sum(xs) / N
            var = sum((v - mean) ** 2 for v in xs) / N
            dl = dsqrt(var + f32_to_fraction(eps))
            assert list(yl[i]) == [round_f16(to_dec((xs[j] - mean) * ws[j]) / dl + to_dec(bs[j]))
                                   for j in range(N)]
            n2 = dsqrt(sum(v * v for v in xs))
            assert list(y2[i]) == [round_f16(to_dec(xs[j]) / n2) for j in range(N)]
        assert np.array_equal(ya, oracle.rmsnorm(h, w, eps, f16=True))


def test_f16_constant_row_closed_form():
    N = 40
    for c in (1.0, -3.5, 1e-3):
        cb = np.array([c], dtype=np.float16).view(np.uint16)[0]
        x = np.full((1, N), cb, dtype=np.uint16)
        w = np.array(np.linspace(0.5, 2, N), dtype=np.float16).view(np.uint16)
        y = oracle.rmsnorm(x, w, 1e-6, f16=True)[0]
        cq = Fraction(float(np.uint16(cb).view(np.float16)))
        den = dsqrt(cq * cq + f32_to_fraction(1e-6))
        want = [round_f16(to_dec(cq * Fraction(float(np.uint16(wj).view(np.float16)))) / den)
                for wj in w]
        assert list(y) == want
