"""GPU parity: the workspace forms (dynamic unit order on the row ring).

With a workspace the persistent row schedule (RN_SCHED_PERSIST_BULK) takes
about 70% of each CTA's units in the fixed order and the rest from a counter
in the workspace, for launches of six units (R rows each) a CTA and more.
Which CTA computes a row must not change its result, so every output is
compared with the oracle and with the fixed order bit for bit, and the
workspace must be zero again after every call, also after a call whose waits
ran out.  Most cases below have six units a CTA or more; a few stay under
it.  Operations: RMSNorm, L2Norm, the fused add and LayerNorm ("[Inductor]
Codegen Gluon", sections 3.1-3.3; "TorchInductor" sections 14.12.2, 14.27).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, norm_bias, rmsnorm_inputs
from tests.gpu_util import require_gpu
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

BULK = binding.RN_SCHED_PERSIST_BULK


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def ws_zero(ws: torch.Tensor) -> bool:
    torch.cuda.synchronize()
    return int(ws.count_nonzero()) == 0


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


# (M, N, debug_flags): many ring wraps with a ragged last unit, forced stage
# counts, two CTAs an SM, generic widths (all six units a CTA and more), then
# launches under the threshold and fewer rows than CTAs
ROW_CASES = [(9001, 1024, 0), (6007, 4096, 3 << 8), (997, 16384, 0), (4001, 8192, 2 << 4),
             (4001, 5120, 0), (3001, 20480, 0), (8001, 3072, 0), (9001, 2048, 4 << 8),
             (300, 32768, 0), (7, 4096, 0), (1000, 2048, 0)]


@pytest.mark.parametrize("M,N,flags", ROW_CASES)
def test_rmsnorm_ring_with_workspace(M, N, flags):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=M + N)
    want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
    xd, wd = x.cuda(), w.cuda()
    ws = binding.new_workspace()
    y_fixed = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK, debug_flags=flags)
    y = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK, debug_flags=flags, workspace=ws)
    assert ws_zero(ws)
    assert_parity(bf16_bits(y), want, f"ws M={M} N={N} flags={flags:#x}")
    assert bits_equal(y, y_fixed)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("op", ["rms", "l2", "add", "ln"])
@pytest.mark.parametrize("M,N", [(6007, 4096), (4001, 8192), (4001, 5120), (1201, 16384)])
def test_other_row_ops_with_workspace(op, M, N, dtype):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=M * 3 + N, dtype=dtype)
    f16 = dtype == torch.float16
    fmt = "f16" if f16 else "bf16"
    xd, wd = x.cuda(), w.cuda()
    ws = binding.new_workspace()
    if op == "rms":
        want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6, f16=f16)
        y0 = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK)
        y = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK, workspace=ws)
    elif op == "l2":
        want = oracle.l2norm(bf16_bits(x), 1e-12, f16=f16)
        y0 = binding.l2norm_fwd(xd, 1e-12, schedule=BULK)
        y = binding.l2norm_fwd(xd, 1e-12, schedule=BULK, workspace=ws)
    elif op == "ln":
        b = norm_bias(N, seed=N, dtype=dtype)
        want = oracle.layernorm(bf16_bits(x), bf16_bits(w), bf16_bits(b), 1e-5, f16=f16)
        y0 = binding.layernorm_fwd(xd, wd, b.cuda(), 1e-5, schedule=BULK)
        y = binding.layernorm_fwd(xd, wd, b.cuda(), 1e-5, schedule=BULK, workspace=ws)
    else:
        r = (rmsnorm_inputs(M, N, seed=N + 5, dtype=torch.float32)[0] * 0.5).to(dtype)
        h_want, want = oracle.add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6, f16=f16)
        h0, y0 = binding.add_rmsnorm_fwd(xd, r.cuda(), wd, 1e-6, schedule=BULK)
        h, y = binding.add_rmsnorm_fwd(xd, r.cuda(), wd, 1e-6, schedule=BULK, workspace=ws)
        assert np.array_equal(bf16_bits(h), h_want)
        assert bits_equal(h, h0)
    assert ws_zero(ws)
    assert_parity(bf16_bits(y), want, f"ws {op} M={M} N={N} {dtype}", fmt=fmt)
    assert bits_equal(y, y0)


def test_schedules_without_a_ring_ignore_the_workspace():
    # one warp per row and one CTA per row never touch it
    ws = binding.new_workspace()
    for M, N, sched in [(4096, 1024, binding.RN_SCHED_WARP_ROW), (64, 4096, binding.RN_SCHED_CTA_ROW),
                        (64, 4096, binding.RN_SCHED_AUTO)]:
        x, w = rmsnorm_inputs(M, N, seed=N)
        y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=sched, workspace=ws)
        assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6), "no ring")
    assert ws_zero(ws)


def test_one_workspace_serves_a_stream_of_calls_and_graph_replays():
    # Back-to-back calls of different shapes and ops (programmatic dependent
    # launch overlaps each one's start with its predecessor's end) share one
    # workspace; so do the replays of a captured graph.
    ws = binding.new_workspace()
    cases = []
    for i, (M, N) in enumerate([(3001, 4096), (2003, 8192), (1500, 16384), (4001, 2048)]):
        x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=50 + i)
        cases.append((x.cuda(), w.cuda(), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)))
    outs = [torch.empty_like(c[0]) for c in cases]
    for rep in range(3):
        for (x, w, _), y in zip(cases, outs):
            binding.rmsnorm_fwd(x, w, 1e-6, y, schedule=BULK, workspace=ws)
    assert ws_zero(ws)
    for (_, _, want), y in zip(cases, outs):
        assert_parity(bf16_bits(y), want, "stream of calls")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for (x, w, _), y in zip(cases, outs):  # warm-up outside the capture
            binding.rmsnorm_fwd(x, w, 1e-6, y, schedule=BULK, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (x, w, _), y in zip(cases, outs):
            binding.rmsnorm_fwd(x, w, 1e-6, y, schedule=BULK, workspace=ws)
    for rep in range(4):
        for y in outs:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (_, _, want), y in zip(cases, outs):
            assert_parity(bf16_bits(y), want, f"graph replay {rep}")
        assert ws_zero(ws)


def test_wait_timeout_with_workspace_leaves_it_zero():
    # The ring is told never to issue its copies: the waits run out (2 ms),
    # the status word records it, and the producers still finish the unit
    # counter, so the workspace is zero and the next call is correct.
    binding.device_status(clear=True)
    ws = binding.new_workspace()
    x, w = rmsnorm_inputs(8192, 4096, seed=3)
    xd, wd = x.cuda(), w.cuda()
    binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK, wait_timeout_ns=2_000_000, debug_flags=1,
                        workspace=ws)
    assert binding.device_status(clear=True) & binding.RN_STATUS_WAIT_TIMEOUT
    assert ws_zero(ws)
    y = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=BULK, workspace=ws)
    assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6), "after timeout")
    assert ws_zero(ws)
    assert binding.device_status(clear=True) == 0
