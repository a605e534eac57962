"""The library's host-memory table builder, rope_cos_sin_table_host (CPU only:
it runs on the calling thread and needs no GPU).

The table feeds the rotation of "[pretuned] Optimize fused_qk_norm_rope on
B200" ("Summary"): row p holds cos(p * f_i) then sin(p * f_i), f_i =
theta^(-2i/r).  It is checked here against the same things that pin the
oracle's table (position 0, the unit circle, 60-digit decimals at chosen
entries) and, entry by entry, against the oracle's table itself.
"""
from __future__ import annotations

import ctypes
from decimal import Decimal

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.build import build
from tests.exact import dcos, dec_to_f32, dsin


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def host_table(lib, theta, max_pos, r):
    out = np.full((max_pos, r), np.nan, dtype=np.float32)
    rc = lib.rope_cos_sin_table_host(theta, max_pos, r, out.ctypes.data_as(ctypes.c_void_p))
    assert rc == binding.RN_OK
    return out


@pytest.mark.parametrize("theta,r", [(1e6, 128), (1e6, 64), (1e4, 8)])
def test_matches_the_oracle_table(lib, theta, r):
    # Both evaluate the angle and the trig in fp64 and round once to fp32.
    # They are separate implementations; an fp64 value within an fp64 step of
    # an fp32 rounding midpoint could round either way, so up to one step on
    # a handful of entries is allowed.
    got = host_table(lib, theta, 6000, r)
    want = oracle.rope_cos_sin(theta, 6000, r)
    assert not np.isnan(got).any()
    steps = np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    assert steps.max() <= 1 and np.count_nonzero(steps) <= 4


def test_position_zero_and_unit_circle(lib):
    t = host_table(lib, 1e6, 4096, 128)
    assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)
    c, s = t[:, :64].astype(np.float64), t[:, 64:].astype(np.float64)
    assert np.max(np.abs(c * c + s * s - 1.0)) < 2**-22


@pytest.mark.parametrize("theta,r,p,i", [(10000.0, 4, 1, 0), (10000.0, 4, 1, 1),
                                         (1e6, 128, 131071, 0), (1e6, 128, 131071, 5),
                                         (1e6, 64, 99991, 31), (1e6, 128, 7, 63)])
def test_entries_against_decimal(lib, theta, r, p, i):
    t = host_table(lib, theta, p + 1, r)
    a = Decimal(p) * Decimal(theta) ** (Decimal(-2 * i) / Decimal(r))
    assert t[p, i] == np.float32(dec_to_f32(dcos(a)))
    assert t[p, r // 2 + i] == np.float32(dec_to_f32(dsin(a)))


def test_argument_checks(lib):
    buf = np.zeros(64, dtype=np.float32)
    p = buf.ctypes.data_as(ctypes.c_void_p)
    assert lib.rope_cos_sin_table_host(1e6, 4, 7, p) == binding.RN_ERR_SHAPE
    assert lib.rope_cos_sin_table_host(1e6, 4, 0, p) == binding.RN_ERR_SHAPE
    assert lib.rope_cos_sin_table_host(-1.0, 4, 8, p) == binding.RN_ERR_SHAPE
    assert lib.rope_cos_sin_table_host(1e6, -1, 8, p) == binding.RN_ERR_SHAPE
    assert lib.rope_cos_sin_table_host(1e6, 4, 8, None) == binding.RN_ERR_NULL
    assert lib.rope_cos_sin_table_host(1e6, 0, 8, None) == binding.RN_OK
    odd = ctypes.c_void_p(buf.ctypes.data + 2)
    assert lib.rope_cos_sin_table_host(1e6, 1, 8, odd) == binding.RN_ERR_ALIGN


def test_binding_builds_a_host_tensor(lib):
    t = binding.rope_cos_sin_table(1e6, 300, 64, device="cpu")
    assert t.device.type == "cpu" and t.dtype == torch.float32
    assert np.array_equal(t.numpy(), host_table(lib, 1e6, 300, 64))
    with pytest.raises(TypeError):
        binding.rope_cos_sin_table(1e6, 4, 8, device="cpu", dtype=torch.bfloat16)
