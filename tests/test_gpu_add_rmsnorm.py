"""GPU parity: fused residual add + RMSNorm (CUDA, through the C ABI) against
the fp64 oracle.

Operation: "TorchInductor: from ATen IR to Triton kernel", sections 14.3 and
14.27 (the norm / residual-add chain fused into one kernel): h = bf16(x + r)
and y = rmsnorm(h).  h must match the oracle bit for bit (a single rounding
of an exact sum); y is held to the RMSNorm tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, rmsnorm_inputs
from tests.full_compare import assert_full_parity
from tests.gpu_util import bulk_eligible, canary_intact, padded_empty, require_gpu
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

SCHEDULES = [binding.RN_SCHED_AUTO, binding.RN_SCHED_WARP_ROW, binding.RN_SCHED_CTA_ROW,
             binding.RN_SCHED_PERSIST_BULK]


def eligible(schedule: int, N: int) -> bool:
    if schedule == binding.RN_SCHED_WARP_ROW:
        return N <= 2048
    if schedule == binding.RN_SCHED_PERSIST_BULK:
        return bulk_eligible(N, "add")
    return True


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def inputs(M, N, seed, device="cpu"):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01 if M >= 100 else 0.0, device=device, seed=seed)
    r, _ = rmsnorm_inputs(M, N, device=device, seed=seed + 50)
    r = (r.float() * 0.5).to(torch.bfloat16)
    return x, r, w


SHAPES = [(1, 8), (7, 64), (5, 1000), (33, 2048), (3, 4104), (130, 1024), (300, 4096),
          (17, 8192), (9, 16384), (5, 32768), (2, 65536), (1000, 512), (2311, 4096)]


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", SHAPES)
def test_small_shapes_every_schedule(M, N, schedule):
    x, r, w = inputs(M, N, seed=M + N)
    h_want, y_want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    pad = 64
    hb, h = padded_empty((M, N), torch.bfloat16, pad, 0x7FC5)
    yb, y = padded_empty((M, N), torch.bfloat16, pad, 0x7FC5)
    if not eligible(schedule, N):
        with pytest.raises(binding.RowNormError) as ei:
            binding.add_rmsnorm_fwd(xd, rd, wd, 1e-6, h, y, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    binding.add_rmsnorm_fwd(xd, rd, wd, 1e-6, h, y, schedule=schedule)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(h), h_want), "h = x + r must be bit-exact"
    assert_parity(bf16_bits(y), y_want, f"add M={M} N={N} sched={schedule}")
    assert canary_intact(hb, pad, 0x7FC5) and canary_intact(yb, pad, 0x7FC5)
    assert np.array_equal(bf16_bits(xd), bf16_bits(x)) and np.array_equal(bf16_bits(rd), bf16_bits(r))


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", [(300, 4096), (2311, 8192), (5, 1000)])
def test_in_place_residual_and_output(M, N, schedule):
    # h written over the residual and y over x: the usual in-place update
    if not eligible(schedule, N):
        return
    x, r, w = inputs(M, N, seed=3 * M + N)
    h_want, y_want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-5)
    xd, rd = x.cuda(), r.cuda()
    binding.add_rmsnorm_fwd(xd, rd, w.cuda(), 1e-5, rd, xd, schedule=schedule)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(rd), h_want)
    assert_parity(bf16_bits(xd), y_want, f"in place M={M} N={N} sched={schedule}")


def test_ring_wraps_with_forced_stages():
    for N, M, stages in [(1024, 5003, 2), (4096, 2311, 3), (16384, 997, 2)]:
        x, r, w = inputs(M, N, seed=N + M)
        h_want, y_want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6)
        h, y = binding.add_rmsnorm_fwd(x.cuda(), r.cuda(), w.cuda(), 1e-6,
                                       schedule=binding.RN_SCHED_PERSIST_BULK,
                                       debug_flags=stages << 8)
        assert np.array_equal(bf16_bits(h), h_want)
        assert_parity(bf16_bits(y), y_want, f"ring N={N} M={M} S={stages}")


def test_wait_timeout_reports_status_and_context_survives():
    binding.device_status(clear=True)
    x, r, w = inputs(2, 1024, seed=3)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    binding.add_rmsnorm_fwd(xd, rd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                            wait_timeout_ns=2_000_000, debug_flags=1)
    assert binding.device_status(clear=True) & binding.RN_STATUS_WAIT_TIMEOUT
    h, y = binding.add_rmsnorm_fwd(xd, rd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK)
    h_want, y_want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6)
    assert np.array_equal(bf16_bits(h), h_want)
    assert_parity(bf16_bits(y), y_want, "after timeout")
    assert binding.device_status(clear=True) == 0


@pytest.mark.parametrize("M,N", [(8192, 8192), (32768, 4096), (4096, 16384), (1024, 32768)])
def test_full_size_every_element(M, N):
    x, r, w = inputs(M, N, seed=7, device="cuda")
    h, y = binding.add_rmsnorm_fwd(x, r, w, 1e-6)
    torch.cuda.synchronize()
    xb, rb, wb = bf16_bits(x), bf16_bits(r), bf16_bits(w)
    del x, r
    assert_full_parity(bf16_bits(y), lambda a, e: oracle.add_rmsnorm(xb[a:e], rb[a:e], wb, 1e-6),
                       f"add full size M={M} N={N}", got_h=bf16_bits(h))


@pytest.mark.parametrize("N", [3072, 5120, 12288, 1000])
def test_non_power_of_two_widths_on_the_ring(N):
    M = 2001
    x, r, w = inputs(M, N, seed=N)
    h_want, y_want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6)
    h, y = binding.add_rmsnorm_fwd(x.cuda(), r.cuda(), w.cuda(), 1e-6,
                                   schedule=binding.RN_SCHED_PERSIST_BULK)
    assert np.array_equal(bf16_bits(h), h_want)
    assert_parity(bf16_bits(y), y_want, f"add ring N={N}")
