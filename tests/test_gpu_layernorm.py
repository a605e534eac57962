"""GPU parity: LayerNorm (CUDA, through the C ABI) against the fp64 oracle.

Operation: "TorchInductor: from ATen IR to Triton kernel", section 14.12.2
(var_mean -> add(eps) -> rsqrt -> sub -> mul -> mul(weight) -> add(bias), one
fused kernel) and "[Inductor] Codegen Gluon", section 3.2 (LayerNorm reuses
its input in both the statistics and the normalise pass).  The oracle uses
the plain two-pass mean and biased variance in double.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, norm_bias, rmsnorm_inputs
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
        return bulk_eligible(N, "ln")
    return True


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SHAPES = [(1, 8), (7, 64), (5, 1000), (33, 2048), (3, 4104), (130, 1024), (300, 4096),
          (17, 8192), (9, 16384), (5, 32768), (2, 65536), (1000, 512), (2311, 4096)]


@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", SHAPES)
def test_small_shapes_every_schedule(M, N, schedule, bias):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.02 if M >= 50 else 0.0, seed=M + 2 * N)
    b = norm_bias(N, seed=M + N) if bias else None
    want = oracle.layernorm(bf16_bits(x), bf16_bits(w), None if b is None else bf16_bits(b), 1e-5)
    pad = 64
    yb, y = padded_empty((M, N), torch.bfloat16, pad, 0x7FC7)
    args = (x.cuda(), w.cuda(), None if b is None else b.cuda(), 1e-5, y)
    if not eligible(schedule, N):
        with pytest.raises(binding.RowNormError) as ei:
            binding.layernorm_fwd(*args, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    binding.layernorm_fwd(*args, schedule=schedule)
    torch.cuda.synchronize()
    assert_parity(bf16_bits(y), want, f"ln M={M} N={N} sched={schedule} bias={bias}")
    assert canary_intact(yb, pad, 0x7FC7)


@pytest.mark.parametrize("schedule", SCHEDULES[1:])
def test_constant_row_gives_the_bias_exactly(schedule):
    N = 2048 if schedule == binding.RN_SCHED_WARP_ROW else 4096
    x = torch.full((4, N), 3.25, dtype=torch.bfloat16)
    w = torch.ones(N, dtype=torch.bfloat16)
    b = norm_bias(N, seed=3)
    y = binding.layernorm_fwd(x.cuda(), w.cuda(), b.cuda(), 1e-5, schedule=schedule)
    assert np.array_equal(bf16_bits(y), np.tile(bf16_bits(b), (4, 1)))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shift", [8.0, 1000.0, -300.0])
@pytest.mark.parametrize("schedule", SCHEDULES[1:])
def test_rows_with_a_large_mean(shift, schedule, dtype):
    # Rows far from zero mean take the centred second reduction, which also
    # corrects the fp32 mean (x - m - c): every output is held to the stated
    # bar, with no allowance for the size of the mean.  Widths 8192 (the mean
    # of bf16 rows is then often exact in fp32) and 5120 or 1000 (it is not),
    # and fp16 rows, whose finer steps make the mean's rounding matter more.
    N = {binding.RN_SCHED_WARP_ROW: 2000, binding.RN_SCHED_CTA_ROW: 5120}.get(schedule, 8192)
    M = 96
    g = torch.Generator().manual_seed(11)
    x = (shift + torch.randn(M, N, generator=g) * torch.linspace(0.5, 4.0, M)[:, None]).to(dtype)
    w = rmsnorm_inputs(1, N, seed=5, dtype=dtype)[1]
    b = norm_bias(N, seed=6, dtype=dtype)
    f16 = dtype == torch.float16
    want = oracle.layernorm(bf16_bits(x), bf16_bits(w), bf16_bits(b), 1e-5, f16=f16)
    for n, sched in [(N, schedule)] + ([(5120, schedule)] if schedule == binding.RN_SCHED_PERSIST_BULK else []):
        xs, ws, bs = x[:, :n].contiguous(), w[:n].contiguous(), b[:n].contiguous()
        ref = want if n == N else oracle.layernorm(bf16_bits(xs), bf16_bits(ws), bf16_bits(bs),
                                                   1e-5, f16=f16)
        y = binding.layernorm_fwd(xs.cuda(), ws.cuda(), bs.cuda(), 1e-5, schedule=sched)
        assert_parity(bf16_bits(y), ref, f"ln shift={shift} N={n} sched={sched} {dtype}",
                      fmt="f16" if f16 else "bf16")


def test_wait_timeout_reports_status_and_context_survives():
    binding.device_status(clear=True)
    x, w = rmsnorm_inputs(2, 1024, seed=3)
    xd, wd = x.cuda(), w.cuda()
    binding.layernorm_fwd(xd, wd, None, 1e-5, schedule=binding.RN_SCHED_PERSIST_BULK,
                          wait_timeout_ns=2_000_000, debug_flags=1)
    assert binding.device_status(clear=True) & binding.RN_STATUS_WAIT_TIMEOUT
    y = binding.layernorm_fwd(xd, wd, None, 1e-5, schedule=binding.RN_SCHED_PERSIST_BULK)
    assert_parity(bf16_bits(y), oracle.layernorm(bf16_bits(x), bf16_bits(w), None, 1e-5), "after")
    assert binding.device_status(clear=True) == 0


# Power-of-two widths, and generic ones in each multi-CTA form at sizes where
# every CTA wraps its ring many times: 3072 (96 x 4, 3 CTAs), 5120 (160 x 4,
# 2 CTAs), 6656 (128 x 8 with a fifth of the slots masked), 12288 (the
# two-CTA build at 8 chunks).
@pytest.mark.parametrize("M,N", [(8192, 8192), (32768, 4096), (4096, 16384), (1024, 32768),
                                 (32768, 3072), (16384, 5120), (16384, 6656), (8192, 12288)])
def test_full_size_every_element(M, N):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, device="cuda", seed=9)
    b = norm_bias(N, device="cuda", seed=10)
    y = binding.layernorm_fwd(x, w, b, 1e-5)
    torch.cuda.synchronize()
    xb, wb, bb, got = bf16_bits(x), bf16_bits(w), bf16_bits(b), bf16_bits(y)
    del x, y
    assert_full_parity(got, lambda a, e: (None, oracle.layernorm(xb[a:e], wb, bb, 1e-5)),
                       f"ln full size M={M} N={N}")


# Generic widths take one of several ring layouts: 1, 2, 4 or 8 chunks a
# thread, with two or three CTAs an SM where a layout covers the row with few
# masked chunks (1000, 2560, 3072, 3584, 5120, 6144, 10240; 11776 and 12288 in
# the two-CTA build at 8 chunks), else one CTA with up to 256 consumers (6656,
# 14336).  2001 rows leave a ragged last round.
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("N", [1000, 2560, 3072, 3584, 5120, 6144, 6656, 10240, 11776, 12288,
                               14336])
def test_non_power_of_two_widths_on_the_ring(N, dtype):
    M = 2001
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=N + 1, dtype=dtype)
    b = norm_bias(N, seed=N + 2, dtype=dtype)
    f16 = dtype == torch.float16
    want = oracle.layernorm(bf16_bits(x), bf16_bits(w), bf16_bits(b), 1e-5, f16=f16)
    y = binding.layernorm_fwd(x.cuda(), w.cuda(), b.cuda(), 1e-5,
                              schedule=binding.RN_SCHED_PERSIST_BULK)
    assert_parity(bf16_bits(y), want, f"ln ring N={N} {dtype}", fmt="f16" if f16 else "bf16")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("N", [4096, 8192, 16384])
def test_rows_either_side_of_the_one_pass_bound(N, dtype):
    # The ring takes the variance from one reduction (E[x^2] - mean^2) when
    # mean^2 <= 4 var and falls back to the centred second pass otherwise:
    # rows with mean / std from 0.5 to 3 put units on both sides, and every
    # output must match the oracle either way.
    M = 1200
    g = torch.Generator().manual_seed(N + 7)
    ratio = torch.tensor([0.5, 1.5, 1.99, 2.01, 2.5, 3.0, 0.0, 1.0])
    xf = torch.randn(M, N, generator=g) + ratio[torch.arange(M) % len(ratio)][:, None]
    x = xf.to(dtype)
    w = rmsnorm_inputs(1, N, seed=8, dtype=dtype)[1]
    b = norm_bias(N, seed=9, dtype=dtype)
    f16 = dtype == torch.float16
    want = oracle.layernorm(bf16_bits(x), bf16_bits(w), bf16_bits(b), 1e-5, f16=f16)
    y = binding.layernorm_fwd(x.cuda(), w.cuda(), b.cuda(), 1e-5,
                              schedule=binding.RN_SCHED_PERSIST_BULK)
    assert_parity(bf16_bits(y), want, f"ln one-pass bound N={N} {dtype}",
                  fmt="f16" if f16 else "bf16")
