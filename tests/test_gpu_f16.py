"""GPU parity: the row norms on IEEE fp16 tensors (CUDA, through the C ABI)
against the fp64 oracle in fp16 mode.

"[Inductor] Codegen Gluon", section 3.2 widens the fused norm's eligible
inputs to fp16.  The kernels are the bf16 ones instantiated for fp16: the
same fp32 arithmetic, one rounding to fp16 at each store.  Tolerance: one
fp16 step per element and at most 2^-7 of the elements one step off (the
fp16 bound in tests/parity.py); h = x + r bit for bit.
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
from tests.parity import assert_parity, parity_report

pytestmark = pytest.mark.gpu

F16 = torch.float16
SCHEDULES = [binding.RN_SCHED_AUTO, binding.RN_SCHED_WARP_ROW, binding.RN_SCHED_CTA_ROW,
             binding.RN_SCHED_PERSIST_BULK]
MODE = {"rms": "rms", "l2": "rms", "add": "add", "ln": "ln"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def eligible(op: str, schedule: int, N: int) -> bool:
    if schedule == binding.RN_SCHED_WARP_ROW:
        return N <= (4096 if op in ("rms", "l2") else 2048)
    if schedule == binding.RN_SCHED_PERSIST_BULK:
        return bulk_eligible(N, MODE[op])
    return True


def make(op, M, N, seed, device="cpu"):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01 if M >= 100 else 0.0, device=device,
                          seed=seed, dtype=F16)
    r = b = None
    if op == "add":
        r = (rmsnorm_inputs(M, N, device=device, seed=seed + 50, dtype=torch.float32)[0]
             * 0.5).to(F16)
    if op == "ln":
        b = norm_bias(N, device=device, seed=seed + 7, dtype=F16)
    return x, r, w, b


def want(op, x, r, w, b, eps):
    """(h or None, y) from the oracle on host copies."""
    xb, wb = bf16_bits(x), bf16_bits(w)
    if op == "rms":
        return None, oracle.rmsnorm(xb, wb, eps, f16=True)
    if op == "l2":
        return None, oracle.l2norm(xb, eps, f16=True)
    if op == "add":
        return oracle.add_rmsnorm(xb, bf16_bits(r), wb, eps, f16=True)
    return None, oracle.layernorm(xb, wb, None if b is None else bf16_bits(b), eps, f16=True)


def run(op, x, r, w, b, eps, h=None, y=None, **kw):
    if op == "rms":
        return None, binding.rmsnorm_fwd(x, w, eps, y, **kw)
    if op == "l2":
        return None, binding.l2norm_fwd(x, eps, y, **kw)
    if op == "add":
        return binding.add_rmsnorm_fwd(x, r, w, eps, h, y, **kw)
    return None, binding.layernorm_fwd(x, w, b, eps, y, **kw)


def dev(t):
    return None if t is None else t.cuda()


EPS = {"rms": 1e-6, "l2": 1e-12, "add": 1e-6, "ln": 1e-5}
SHAPES = [(1, 8), (7, 64), (5, 1000), (33, 2048), (3, 4104), (130, 1024), (300, 4096),
          (17, 8192), (9, 16384), (5, 32768), (2, 65536), (1000, 512), (2311, 4096)]


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("op", ["rms", "l2", "add", "ln"])
def test_small_shapes_every_schedule(op, M, N, schedule):
    x, r, w, b = make(op, M, N, seed=M + 3 * N)
    eps = EPS[op]
    h_want, y_want = want(op, x, r, w, b, eps)
    pad = 64
    yb, y = padded_empty((M, N), F16, pad, 0x7E11)
    hb, h = padded_empty((M, N), F16, pad, 0x7E11)
    args = (op, dev(x), dev(r), dev(w), dev(b), eps)
    if not eligible(op, schedule, N):
        with pytest.raises(binding.RowNormError) as ei:
            run(*args, h=h if op == "add" else None, y=y, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    run(*args, h=h if op == "add" else None, y=y, schedule=schedule)
    torch.cuda.synchronize()
    assert y.dtype == F16
    if op == "add":
        assert np.array_equal(bf16_bits(h), h_want), "h = x + r must be bit-exact"
        assert canary_intact(hb, pad, 0x7E11)
    assert_parity(bf16_bits(y), y_want, f"f16 {op} M={M} N={N} sched={schedule}", fmt="f16")
    assert canary_intact(yb, pad, 0x7E11)


@pytest.mark.parametrize("op", ["rms", "l2", "add", "ln"])
@pytest.mark.parametrize("N", [3072, 5120, 12288, 1000])
def test_non_power_of_two_widths_on_the_ring(op, N):
    M = 2001
    x, r, w, b = make(op, M, N, seed=N + 11)
    h_want, y_want = want(op, x, r, w, b, EPS[op])
    h, y = run(op, dev(x), dev(r), dev(w), dev(b), EPS[op],
               schedule=binding.RN_SCHED_PERSIST_BULK)
    if op == "add":
        assert np.array_equal(bf16_bits(h), h_want)
    assert_parity(bf16_bits(y), y_want, f"f16 {op} ring N={N}", fmt="f16")


@pytest.mark.parametrize("op", ["rms", "add", "ln"])
@pytest.mark.parametrize("M,N", [(8192, 8192), (32768, 4096), (4096, 16384), (1024, 32768)])
def test_full_size_every_element(op, M, N):
    x, r, w, b = make(op, M, N, seed=7, device="cuda")
    h, y = run(op, x, r, w, b, EPS[op])
    torch.cuda.synchronize()
    xb, wb = bf16_bits(x), bf16_bits(w)
    rb = None if r is None else bf16_bits(r)
    bb = None if b is None else bf16_bits(b)
    eps = EPS[op]

    def rows(a, e):
        if op == "rms":
            return None, oracle.rmsnorm(xb[a:e], wb, eps, f16=True)
        if op == "add":
            return oracle.add_rmsnorm(xb[a:e], rb[a:e], wb, eps, f16=True)
        return None, oracle.layernorm(xb[a:e], wb, bb, eps, f16=True)

    assert_full_parity(bf16_bits(y), rows, f"f16 {op} full size M={M} N={N}", fmt="f16",
                       got_h=None if h is None else bf16_bits(h))


@pytest.mark.parametrize("schedule", SCHEDULES[1:])
def test_overflow_to_infinity_matches(schedule):
    # weights near the fp16 maximum push some outputs past 65504: both sides
    # round them to infinity, every finite output stays within tolerance
    N = 2048 if schedule == binding.RN_SCHED_WARP_ROW else 4096
    x, _ = rmsnorm_inputs(300, N, seed=21, dtype=F16)
    w = torch.full((N,), 30000.0, dtype=F16)
    y_want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6, f16=True)
    assert (np.abs(y_want.view(np.float16)) == np.inf).sum() > 100
    y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=schedule)
    got = bf16_bits(y)
    assert_parity(got, y_want, f"f16 overflow sched={schedule}", fmt="f16")
    inf_g = np.isinf(got.view(np.float16))
    inf_w = np.isinf(y_want.view(np.float16))
    assert (inf_g != inf_w).sum() <= 2  # only at the 65504 / 65520 boundary


@pytest.mark.parametrize("schedule", SCHEDULES[1:])
def test_subnormal_outputs(schedule):
    # weights of 2^-20 put every output among fp16 subnormals (step 2^-24)
    N = 2048 if schedule == binding.RN_SCHED_WARP_ROW else 4096
    x, _ = rmsnorm_inputs(300, N, seed=23, dtype=F16)
    w = torch.full((N,), 2.0**-20, dtype=F16)
    y_want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6, f16=True)
    y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=schedule)
    rep = parity_report(bf16_bits(y), y_want, fmt="f16")
    assert rep["max_ulp"] <= 1 and rep["one_ulp_frac"] <= 2.0**-7, rep
    assert np.count_nonzero(y_want & 0x7C00) == 0  # all subnormal or zero


@pytest.mark.parametrize("op", ["rms", "add", "ln"])
def test_in_place(op):
    # y written over x (and h over the residual for the fused add)
    M, N = 300, 4096
    x, r, w, b = make(op, M, N, seed=31)
    h_want, y_want = want(op, x, r, w, b, EPS[op])
    xd, rd = dev(x), dev(r)
    run(op, xd, rd, dev(w), dev(b), EPS[op], h=rd, y=xd)
    torch.cuda.synchronize()
    if op == "add":
        assert np.array_equal(bf16_bits(rd), h_want)
    assert_parity(bf16_bits(xd), y_want, f"f16 {op} in place", fmt="f16")


def test_wait_timeout_in_the_f16_kernels_reports_status():
    binding.device_status(clear=True)
    x, _, w, _ = make("rms", 2, 1024, seed=3)
    xd, wd = x.cuda(), w.cuda()
    binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                        wait_timeout_ns=2_000_000, debug_flags=1)
    assert binding.device_status(clear=True) & binding.RN_STATUS_WAIT_TIMEOUT
    y = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK)
    assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6, f16=True),
                  "after", fmt="f16")
    assert binding.device_status(clear=True) == 0


def test_schedule_choice_does_not_depend_on_the_format():
    for M, N in [(8, 1024), (8192, 2048), (32768, 4096), (4096, 5120), (64, 65536)]:
        assert binding.row_norm_select_schedule(binding.RN_OP_RMSNORM, M, N) == \
            binding.rmsnorm_select_schedule(M, N)
        assert binding.row_norm_select_schedule(binding.RN_OP_ADD_RMSNORM, M, N) == \
            binding.add_rmsnorm_select_schedule(M, N)
        assert binding.row_norm_select_schedule(binding.RN_OP_LAYERNORM, M, N) == \
            binding.layernorm_select_schedule(M, N)


@pytest.mark.parametrize("op", ["rms", "ln", "l2", "add"])
def test_subnormal_inputs(op):
    # x ~ 1e-6 lies among fp16 subnormals (the smallest normal is 2^-14 =
    # 6.1e-5): the kernels widen them exactly, so with a tiny eps the rows
    # normalise to O(1) outputs that must match the oracle
    M, N = 600, 4096
    g = torch.Generator().manual_seed(61)
    x = (torch.randn(M, N, generator=g) * 1e-6).to(F16)
    assert (bf16_bits(x) & 0x7C00 == 0).mean() > 0.9  # mostly subnormal
    w = rmsnorm_inputs(1, N, seed=62, dtype=F16)[1]
    b = norm_bias(N, seed=63, dtype=F16)
    r = (torch.randn(M, N, generator=g) * 1e-6).to(F16)
    eps = {"rms": 1e-14, "ln": 1e-14, "l2": 1e-12, "add": 1e-14}[op]
    xb, wb = bf16_bits(x), bf16_bits(w)
    if op == "rms":
        want = oracle.rmsnorm(xb, wb, eps, f16=True)
        got = binding.rmsnorm_fwd(x.cuda(), w.cuda(), eps)
    elif op == "ln":
        want = oracle.layernorm(xb, wb, bf16_bits(b), eps, f16=True)
        got = binding.layernorm_fwd(x.cuda(), w.cuda(), b.cuda(), eps)
    elif op == "l2":
        want = oracle.l2norm(xb, eps, f16=True)
        got = binding.l2norm_fwd(x.cuda(), eps)
    else:
        h_want, want = oracle.add_rmsnorm(xb, bf16_bits(r), wb, eps, f16=True)
        h, got = binding.add_rmsnorm_fwd(x.cuda(), r.cuda(), w.cuda(), eps)
        assert np.array_equal(bf16_bits(h), h_want)
    assert_parity(bf16_bits(got), want, f"f16 subnormal inputs {op}", fmt="f16")
