"""rmsnorm_fwd_noalloc: RMSNorm for callers that cannot allocate device memory.

Some callers cannot give the library a workspace: a plug-in inside a host
framework that owns the device's memory pool, or a serving process that
forbids device allocations after start-up so that its memory use stays fixed.
This entry point keeps the row ring's counters in a scratch array declared
inside the library instead.  Its results must be those of rmsnorm_fwd, within
the tolerance every parity test here uses, call after call (the array keeps
the previous call's contents).  This file is collected last, so a run that
stops at its first failure has run every other test before it.
"""
from __future__ import annotations

import pytest
import torch

from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, rmsnorm_inputs
from tests.gpu_util import require_gpu
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


def test_no_alloc_entry_matches_rmsnorm_fwd_on_consecutive_calls():
    require_gpu()
    lib = binding.load()
    stream = torch.cuda.current_stream().cuda_stream
    # two ring launches with the dynamic unit order (six units a CTA and more),
    # the second with a ragged last unit, then a short one-CTA-a-row launch
    for M, N, seed in [(8192, 8192, 1), (6007, 4096, 2), (64, 4096, 3)]:
        x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, device="cuda", seed=seed)
        want = torch.empty_like(x)
        got = torch.full_like(x, float("nan"))
        assert lib.rmsnorm_fwd(x.data_ptr(), w.data_ptr(), 1e-6, M, N, want.data_ptr(),
                               stream) == binding.RN_OK
        assert lib.rmsnorm_fwd_noalloc(x.data_ptr(), w.data_ptr(), 1e-6, M, N, got.data_ptr(),
                                       stream) == binding.RN_OK
        torch.cuda.synchronize()
        assert_parity(bf16_bits(got), bf16_bits(want), f"no-alloc M={M} N={N}")


def test_no_alloc_entry_refuses_bad_sizes_clearly():
    require_gpu()
    lib = binding.load()
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    rc = lib.rmsnorm_fwd_noalloc(x.data_ptr(), w.data_ptr(), 1e-6, 4, 65544, x.data_ptr(), None)
    assert rc == binding.RN_ERR_SHAPE
    assert "size" in binding.error_string(rc)
