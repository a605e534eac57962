"""Stream order with programmatic dependent launch (GPU).

Every kernel may be scheduled while the previous launch on the stream is
still finishing; it must wait for that launch before touching memory.  A
chain in which each call consumes the previous call's output (back to back,
and interleaved with torch's own kernels) therefore has to give exactly what
the oracle gives applied step by step.  A kernel that read its input early
would see stale data here.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, bf16_from_bits, norm_bias, rmsnorm_inputs
from tests.gpu_util import require_gpu
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("M,N", [(4096, 4096), (300, 8192), (20000, 2048)])
def test_dependent_chain_matches_the_oracle_step_by_step(M, N):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=M + N)
    b = norm_bias(N, seed=5)
    xd, wd, bd = x.cuda(), w.cuda(), b.cuda()
    y1 = torch.empty_like(xd)
    y2 = torch.empty_like(xd)
    y3 = torch.empty_like(xd)
    h = torch.empty_like(xd)
    y4 = torch.empty_like(xd)
    for _ in range(3):  # several rounds: each round's launches follow the previous round's
        binding.rmsnorm_fwd(xd, wd, 1e-6, y1)
        binding.rmsnorm_fwd(y1, wd, 1e-6, y2)          # reads y1 right after it is written
        binding.layernorm_fwd(y2, wd, bd, 1e-5, y3)    # reads y2
        binding.add_rmsnorm_fwd(y3, y1, wd, 1e-6, h, y4)
    torch.cuda.synchronize()
    wb, bb = bf16_bits(w), bf16_bits(b)
    g1, g2, g3, gh, g4 = (bf16_bits(t) for t in (y1, y2, y3, h, y4))
    assert_parity(g1, oracle.rmsnorm(bf16_bits(x), wb, 1e-6), "step 1")
    # each later step is checked on the GPU's own previous output, so one
    # step's legitimate rounding cannot cascade into the next comparison
    assert_parity(g2, oracle.rmsnorm(g1, wb, 1e-6), "step 2")
    assert_parity(g3, oracle.layernorm(g2, wb, bb, 1e-5), "step 3")
    h_want, y_want = oracle.add_rmsnorm(g3, g1, wb, 1e-6)
    assert np.array_equal(gh, h_want)
    assert_parity(g4, y_want, "step 4")


def test_interleaved_with_torch_kernels():
    M, N = 8192, 4096
    x, w = rmsnorm_inputs(M, N, seed=3)
    xd, wd = x.cuda(), w.cuda()
    y = torch.empty_like(xd)
    binding.rmsnorm_fwd(xd, wd, 1e-6, y)
    xd.mul_(2.0)                          # torch kernel between two of ours
    y2 = binding.rmsnorm_fwd(xd, wd, 1e-6)
    z = (y2.float() * 0.5).to(torch.bfloat16)   # torch kernel reading our output
    torch.cuda.synchronize()
    x2 = bf16_bits((x.float() * 2.0).to(torch.bfloat16))
    assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6), "before")
    want2 = oracle.rmsnorm(x2, bf16_bits(w), 1e-6)
    assert_parity(bf16_bits(y2), want2, "after a torch kernel")
    z_want = (bf16_from_bits(bf16_bits(y2)).float() * 0.5).to(torch.bfloat16)
    assert torch.equal(z.cpu().view(torch.int16), z_want.view(torch.int16))
