"""GPU parity: rmsnorm_fwd (CUDA, through the C ABI) against the fp64 oracle.

RMSNorm: "[Inductor] Codegen Gluon", section 3.1.  Sizes: small shapes that
span several tiles with ragged tails for every schedule (full comparison),
then the measured workloads at full size in the launch configuration the
bench times (every element against the oracle, the rows split over the host
cores).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, rmsnorm_inputs
from tests.exact import bits_to_f64
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


SMALL_SHAPES = [(1, 8), (3, 8), (7, 64), (5, 1000), (33, 2048), (3, 4104), (130, 1024),
                (300, 4096), (17, 8192), (9, 16384), (5, 32768), (2, 65536), (1000, 512),
                (157, 3072), (611, 2048), (45, 2056), (61, 2560), (29, 3584)]


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("M,N", SMALL_SHAPES)
def test_small_shapes_every_schedule(M, N, schedule):
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.05 if M >= 20 else 0.0, seed=M * 7 + N)
    want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
    xd, wd = x.cuda(), w.cuda()
    pad = 64
    buf, y = padded_empty((M, N), torch.bfloat16, pad, 0x7FC1)
    if not eligible(schedule, N):
        with pytest.raises(binding.RowNormError) as ei:
            binding.rmsnorm_fwd(xd, wd, 1e-6, y, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    binding.rmsnorm_fwd(xd, wd, 1e-6, y, schedule=schedule)
    torch.cuda.synchronize()
    assert_parity(bf16_bits(y), want, f"M={M} N={N} sched={schedule}")
    assert canary_intact(buf, pad, 0x7FC1), "write outside y"
    assert np.array_equal(bf16_bits(xd), bf16_bits(x)), "x modified"


def test_persistent_ring_wraps_many_times_with_ragged_split():
    # Many more units than stages, M not a multiple of the grid or of R.
    for N, M, stages in [(1024, 5003, 2), (4096, 2311, 3), (16384, 997, 2)]:
        x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=N + M)
        want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
        y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                                debug_flags=stages << 8)
        assert_parity(bf16_bits(y), want, f"ring N={N} M={M} S={stages}")


def test_two_ctas_per_sm_variant():
    # two co-resident persistent CTAs per SM, each with a two-stage ring
    x, w = rmsnorm_inputs(1201, 8192, seed=5)
    want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
    y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                            debug_flags=2 << 4)
    assert_parity(bf16_bits(y), want, "2 CTAs/SM")


@pytest.mark.parametrize("N,ctas", [(16384, 8), (32768, 4), (5120, 15)])
def test_more_ctas_per_sm_than_fit_are_clamped(N, ctas):
    # A request for more CTAs an SM than registers and shared memory allow is
    # clamped to what fits (otherwise the rest would queue as a second wave);
    # the rows still all come out right, ragged last round included.
    M = 1301
    x, w = rmsnorm_inputs(M, N, seed=N + ctas)
    want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
    y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                            debug_flags=ctas << 4)
    assert_parity(bf16_bits(y), want, f"ring N={N} asking {ctas} CTAs/SM")


def exact_rmsnorm(x, w, eps):
    """Unrounded RMSNorm outputs in float64 (the oracle's row scale)."""
    xb, wb = bf16_bits(x), bf16_bits(w)
    rs = oracle.rms_rstd(xb, eps)
    return bits_to_f64(xb) * rs[:, None] * bits_to_f64(wb)[None, :]


def test_special_rows():
    # Degenerate rows, checked element by element: a one-step difference is
    # allowed only where the exact value sits at a rounding midpoint within
    # the fp32 error bound.  Seed 253 gives a row whose fp32 scale puts one
    # bf16 mantissa 2^-24 from a midpoint (26 elements move together on the
    # CTA-per-row schedule at eps 1e-30): correct arithmetic that a fraction
    # budget over 6 rows would misjudge.
    N = 4096
    g = torch.Generator().manual_seed(253)
    x = torch.zeros(6, N, dtype=torch.bfloat16)
    x[1] = 3.0                       # constant row
    x[2, 17] = -7.5                  # one-hot row
    x[3] = torch.randn(N, generator=g) * 1e-3     # tiny values: eps dominates
    x[4] = torch.randn(N, generator=g) * 1e3
    x[5, ::2] = 1.0
    w = torch.ones(N, dtype=torch.bfloat16)
    for eps in (1e-6, 1e-5, 0.0 + 1e-30):
        want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), eps)
        exact = exact_rmsnorm(x, w, eps)
        for sched in SCHEDULES[1:]:
            if not eligible(sched, N):
                continue
            y = binding.rmsnorm_fwd(x.cuda(), w.cuda(), eps, schedule=sched)
            got = bf16_bits(y)
            assert_parity(got, want, f"special eps={eps} sched={sched}", exact=exact)
            assert np.all(got[0] == 0)  # zero row stays zero


def test_empty_and_errors():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    assert binding.rmsnorm_fwd(x, w, 1e-6).shape == (0, 64)
    with pytest.raises(binding.RowNormError):
        xx = torch.ones(4, 12, dtype=torch.bfloat16, device="cuda")
        binding.rmsnorm_fwd(xx, torch.ones(12, dtype=torch.bfloat16, device="cuda"), 1e-6)
    with pytest.raises(binding.RowNormError) as ei:
        binding.rmsnorm_fwd(torch.ones(2, 7, dtype=torch.bfloat16, device="cuda"),
                            torch.ones(7, dtype=torch.bfloat16, device="cuda"), 1e-6)
    assert ei.value.code == binding.RN_ERR_SHAPE


def test_wait_timeout_reports_status_and_context_survives():
    # The persistent schedule is told never to issue its copies, so its
    # bounded waits run out (2 ms): the kernel must record the timeout in the
    # status word and return, leaving the context usable.
    binding.device_status(clear=True)
    x, w = rmsnorm_inputs(2, 1024, seed=3)
    xd, wd = x.cuda(), w.cuda()
    binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK,
                        wait_timeout_ns=2_000_000, debug_flags=1)
    st = binding.device_status(clear=True)
    assert st & binding.RN_STATUS_WAIT_TIMEOUT
    y = binding.rmsnorm_fwd(xd, wd, 1e-6, schedule=binding.RN_SCHED_PERSIST_BULK)
    assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6), "after timeout")
    assert binding.device_status(clear=True) == 0


# ---------------------------------------------------------------------------
# Full-size workloads, auto schedule (what the bench launches)
# ---------------------------------------------------------------------------

def _check_full_size(M, N, eps, outlier_frac, seed=0, schedule=binding.RN_SCHED_AUTO):
    """The launch the bench times (with a workspace: the dynamic unit order),
    every element against the oracle.  The plain form gives the same bits
    when it takes the same schedule (the unit order and the stage count do
    not change a row's arithmetic); where it takes another (RMSNorm 4096 wide
    over many rows: one warp per row), its output is compared in full too."""
    x, w = rmsnorm_inputs(M, N, outlier_frac=outlier_frac, device="cuda", seed=seed)
    ws = binding.new_workspace()
    y = binding.rmsnorm_fwd(x, w, eps, workspace=ws, schedule=schedule)
    y_plain = binding.rmsnorm_fwd(x, w, eps, schedule=schedule)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    same = schedule != binding.RN_SCHED_AUTO or \
        binding.rmsnorm_select_schedule(M, N, workspace=True) == binding.rmsnorm_select_schedule(M, N)
    if same:
        assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))
        outs = [("", bf16_bits(y))]
    else:
        outs = [(" workspace", bf16_bits(y)), (" plain", bf16_bits(y_plain))]
    xb, wb = bf16_bits(x), bf16_bits(w)
    del x, y, y_plain
    for tag, got in outs:
        assert_full_parity(got, lambda a, b: (None, oracle.rmsnorm(xb[a:b], wb, eps)),
                           f"full size M={M} N={N}{tag}")


def test_latency_config_full():
    # 64 x 4096: small enough to compare every element with the oracle
    x, w = rmsnorm_inputs(64, 4096, device="cuda", seed=0)
    y = binding.rmsnorm_fwd(x, w, 1e-6)
    assert_parity(bf16_bits(y), oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6), "64x4096")


@pytest.mark.parametrize("M", [4096, 8192, 16384, 32768])
@pytest.mark.parametrize("N", [4096, 8192, 16384])
def test_sweep_full_size(M, N):
    _check_full_size(M, N, 1e-6, 0.01)


@pytest.mark.parametrize("M,N", [(24576, 3072), (20480, 3584), (32768, 2560)])
def test_many_rows_up_to_4096_wide_take_one_warp_a_row(M, N):
    # 128 rows an SM and more, 2049..4095 wide: one warp per row, 12 or 16
    # chunks a lane (masked past the row end), chosen automatically
    assert binding.rmsnorm_select_schedule(M, N) == binding.RN_SCHED_WARP_ROW
    _check_full_size(M, N, 1e-6, 0.01)


def test_many_rows_4096_wide_ring_and_one_warp_a_row():
    # 4096 wide: RMSNorm with a workspace takes the four-stage ring at every
    # row count, without one one warp per row from 128 rows an SM; L2Norm one
    # warp per row from 12 rows an SM either way
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M in (8192, 32768, 131072):
        assert binding.rmsnorm_select_schedule(M, 4096, workspace=True) == \
            binding.RN_SCHED_PERSIST_BULK
    assert binding.rmsnorm_select_schedule(128 * sms - 8, 4096) == binding.RN_SCHED_PERSIST_BULK
    assert binding.rmsnorm_select_schedule(128 * sms, 4096) == binding.RN_SCHED_WARP_ROW
    for ws in (False, True):
        assert binding.row_norm_select_schedule(binding.RN_OP_L2NORM, 12 * sms, 4096,
                                                workspace=ws) == binding.RN_SCHED_WARP_ROW
    _check_full_size(131072, 4096, 1e-6, 0.01)


@pytest.mark.parametrize("M", [1024, 4096, 8192])
def test_wide_rows_full_size(M):
    _check_full_size(M, 32768, 1e-5, 0.0)


@pytest.mark.parametrize("N", [3072, 5120, 6656, 12288, 20480, 4104, 1000])
def test_non_power_of_two_widths_on_the_ring(N):
    # common hidden sizes that are not powers of two: the masked generic ring
    M = 3001
    x, w = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=N)
    want = oracle.rmsnorm(bf16_bits(x), bf16_bits(w), 1e-6)
    pad = 64
    buf, y = padded_empty((M, N), torch.bfloat16, pad, 0x7FC1)
    binding.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6, y, schedule=binding.RN_SCHED_PERSIST_BULK)
    torch.cuda.synchronize()
    assert_parity(bf16_bits(y), want, f"ring N={N}")
    assert canary_intact(buf, pad, 0x7FC1)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_rows_with_extreme_scales(schedule):
    # Rows from 2^-55 to 2^50 in magnitude (with eps = 0 the tiny rows get
    # scales up to 2^55), and a weight vector holding 2^70: every output must
    # still agree with the oracle.
    N, M = 4096, 2000
    g = torch.Generator().manual_seed(41)
    x = torch.randn(M, N, generator=g)
    scale = torch.tensor([1.0, 2.0**50, 2.0**-55, 2.0**35, 2.0**-35, 2.0**45, 2.0**-38, 1.0])
    x = (x * scale[torch.arange(M) % len(scale)][:, None]).to(torch.bfloat16)
    w = rmsnorm_inputs(1, N, seed=42)[1]
    w_big = w.clone()
    w_big[777] = 2.0**70
    for ww in (w, w_big):
        for eps in (0.0, 1e-6):
            want = oracle.rmsnorm(bf16_bits(x), bf16_bits(ww), eps)
            if not eligible(schedule, N):
                continue
            y = binding.rmsnorm_fwd(x.cuda(), ww.cuda(), eps, schedule=schedule)
            assert_parity(bf16_bits(y), want, f"extreme rows eps={eps} sched={schedule}",
                          exact=exact_rmsnorm(x, ww, eps))
