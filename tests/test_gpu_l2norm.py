"""GPU parity: L2Norm (CUDA, through the C ABI) against the fp64 oracle.

Operation: "[Inductor] Codegen Gluon", section 3.2 (L2Norm: a single
reduction, then a scale by the inverse norm); y = x / max(||x||_2, eps).
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
        return N <= 4096  # RMSNorm and L2Norm take one warp per row up to 4096 wide
    if schedule == binding.RN_SCHED_PERSIST_BULK:
        return bulk_eligible(N, "rms")
    return True


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SHAPES = [(1, 8), (7, 64), (5, 1000), (33, 2048), (3, 4104), (130, 1024), (300, 4096),
          (17, 8192), (9, 16384), (5, 32768), (2, 65536), (2311, 4096)]


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", SHAPES)
def test_small_shapes_every_schedule(M, N, schedule):
    x, _ = rmsnorm_inputs(M, N, outlier_frac=0.05 if M >= 20 else 0.0, seed=M + 5 * N)
    want = oracle.l2norm(bf16_bits(x), 1e-12)
    pad = 64
    yb, y = padded_empty((M, N), torch.bfloat16, pad, 0x7FC9)
    if not eligible(schedule, N):
        with pytest.raises(binding.RowNormError) as ei:
            binding.l2norm_fwd(x.cuda(), 1e-12, y, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    binding.l2norm_fwd(x.cuda(), 1e-12, y, schedule=schedule)
    torch.cuda.synchronize()
    assert_parity(bf16_bits(y), want, f"l2 M={M} N={N} sched={schedule}")
    assert canary_intact(yb, pad, 0x7FC9)


@pytest.mark.parametrize("schedule", SCHEDULES[1:])
def test_rows_below_eps_and_zero_rows(schedule):
    N = 2048 if schedule == binding.RN_SCHED_WARP_ROW else 4096
    x = torch.zeros(4, N, dtype=torch.bfloat16)
    x[1] = 2.0**-20                    # norm below eps: divided by eps
    x[2, 7] = -3.0                     # one-hot: -1 at 7
    x[3] = torch.randn(N) * 1e-2
    eps = 1e-3
    y = binding.l2norm_fwd(x.cuda(), eps, schedule=schedule)
    assert_parity(bf16_bits(y), oracle.l2norm(bf16_bits(x), eps), f"l2 special sched={schedule}")
    assert np.all(bf16_bits(y)[0] == 0)


@pytest.mark.parametrize("M,N", [(8192, 8192), (32768, 4096), (1024, 32768)])
def test_full_size_every_element(M, N):
    x, _ = rmsnorm_inputs(M, N, outlier_frac=0.01, device="cuda", seed=13)
    y = binding.l2norm_fwd(x, 1e-12)
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    del x
    assert_full_parity(bf16_bits(y), lambda a, e: (None, oracle.l2norm(xb[a:e], 1e-12)),
                       f"l2 full size M={M} N={N}")
