"""GPU parity: fused Q/K RMSNorm + neox RoPE (CUDA, through the C ABI)
against the fp64 oracle, and the device cos/sin table builder.

Operation: "[pretuned] Optimize fused_qk_norm_rope on B200", section
"Summary".  Every head layout the library supports is checked on small
token counts under every schedule; the measured workloads (32 query and 8
key/value heads of 128, full and half rotary, up to 16384 tokens) are
compared element by element in full.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, qkv_inputs
from tests.gpu_util import (canary_intact, oracle_table, oracle_table_bf16, padded_empty,
                            require_gpu)
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

QK_SCHEDULES = [binding.RN_QK_AUTO, binding.RN_QK_HEAD_PER_WARP, binding.RN_QK_TWO_HEADS,
                binding.RN_QK_FOUR_HEADS, binding.RN_QK_PERSISTENT, binding.RN_QK_BULK,
                binding.RN_QK_PAIRS]
# the ring does not take D 64 with rotary 16 (one element a lane per half)
NOT_64_16 = (binding.RN_QK_BULK,)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_case(T, Hq, Hkv, D, r, *, positions="arange", max_pos=None, theta=1e6, eps=1e-6,
             schedule=binding.RN_QK_AUTO, device_inputs=False, seed=0, debug_flags=0,
             style=binding.RN_ROPE_NEOX, bf16_table=False):
    max_pos = max_pos or max(T, 1)
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions=positions, max_pos=max_pos,
                                  device="cuda" if device_inputs else "cpu", seed=seed)
    if bf16_table:
        # the oracle reads the bf16 entries widened to fp32, as the kernels do
        dev_table, table = oracle_table_bf16(theta, max_pos, r)
    else:
        table = oracle_table(theta, max_pos, r)
        dev_table = torch.from_numpy(table).cuda()
    want = oracle.qk_norm_rope(bf16_bits(qkv), bf16_bits(wq), bf16_bits(wk), table,
                               pos.cpu().numpy(), Hq, Hkv, D, r, eps, style=style)
    pad = 128
    buf, q = padded_empty(tuple(qkv.shape), torch.bfloat16, pad, 0x7FC3)
    q.copy_(qkv)
    if style == binding.RN_ROPE_NEOX:
        binding.qk_norm_rope_fwd(q, wq.cuda(), wk.cuda(), dev_table, pos.cuda(), Hq, Hkv, D, r,
                                 eps, schedule=schedule, debug_flags=debug_flags)
    else:
        binding.qk_norm_rope_fwd_ex(q, wq.cuda(), wk.cuda(), dev_table, pos.cuda(), Hq, Hkv, D,
                                    r, eps, rope_style=style, schedule=schedule,
                                    debug_flags=debug_flags)
    torch.cuda.synchronize()
    got = bf16_bits(q)
    assert canary_intact(buf, pad, 0x7FC3), "write outside qkv"
    # value heads untouched, bit for bit
    W = (Hq + 2 * Hkv) * D
    v0 = (Hq + Hkv) * D
    assert np.array_equal(got.reshape(T, W)[:, v0:], bf16_bits(qkv).reshape(T, W)[:, v0:])
    return got, want


LAYOUTS = [(64, 64), (64, 32), (64, 16), (128, 128), (128, 64), (128, 32),
           (256, 256), (256, 128), (256, 64)]


@pytest.mark.parametrize("schedule", QK_SCHEDULES)
@pytest.mark.parametrize("D,r", LAYOUTS)
def test_layouts_every_schedule(D, r, schedule):
    if schedule in NOT_64_16 and (D, r) == (64, 16):
        # one element per lane per rotary half: only the warp schedules take it
        with pytest.raises(binding.RowNormError) as ei:
            run_case(5, 4, 2, D, r, positions="uniform", max_pos=97, schedule=schedule)
        assert ei.value.code == binding.RN_ERR_SHAPE
        return
    got, want = run_case(5, 4, 2, D, r, positions="uniform", max_pos=97, schedule=schedule,
                         seed=D + r)
    assert_parity(got, want, f"D={D} r={r} sched={schedule}")


@pytest.mark.parametrize("schedule", [binding.RN_QK_AUTO, binding.RN_QK_BULK, binding.RN_QK_PAIRS])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (1, 0), (0, 2), (7, 3), (1, 1), (64, 0)])
@pytest.mark.parametrize("T", [1, 2, 3, 33, 1000])
def test_head_counts_ragged(T, Hq, Hkv, schedule):
    got, want = run_case(T, Hq, Hkv, 128, 128, positions="uniform", max_pos=4096,
                         seed=T * 100 + Hq, schedule=schedule)
    assert_parity(got, want, f"T={T} Hq={Hq} Hkv={Hkv} sched={schedule}")


@pytest.mark.parametrize("D,r", [lr for lr in LAYOUTS if lr != (64, 16)])
def test_bulk_ring_many_units_every_layout(D, r):
    # thousands of tokens: every CTA wraps its two-stage ring many times and the
    # last round is split unevenly
    got, want = run_case(3001, 8, 2, D, r, positions="uniform", max_pos=9000,
                         schedule=binding.RN_QK_BULK, seed=D * 3 + r)
    assert_parity(got, want, f"bulk D={D} r={r}")
    for stages in (2, 3, 6):
        got, want = run_case(777, 8, 2, D, r, positions="uniform", max_pos=9000,
                             schedule=binding.RN_QK_BULK, seed=stages, debug_flags=stages << 8)
        assert_parity(got, want, f"bulk D={D} r={r} stages={stages}")


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 2), (12, 4), (5, 2)])
@pytest.mark.parametrize("D,r", LAYOUTS)
def test_pairs_many_rounds_every_layout(D, r, Hq, Hkv):
    # Two heads per lane group (4, 8 or 16 lanes a head at D 64, 128, 256).
    # A round covers 16, 8 or 4 consecutive heads: where that divides the
    # normed heads a token, both heads of a group are always one token's;
    # elsewhere (10 or 7 heads a token, 40 at D 64) they straddle two tokens
    # in some rounds, which reads a second cos/sin row.  About 200 000 heads:
    # several rounds a warp on the two-wave grid, the last one ragged.
    T = 200_000 // (Hq + Hkv) + 1
    got, want = run_case(T, Hq, Hkv, D, r, positions="uniform", max_pos=9000,
                         schedule=binding.RN_QK_PAIRS, seed=D * 5 + r + Hq, device_inputs=True)
    assert_parity(got, want, f"pairs D={D} r={r} Hq={Hq} Hkv={Hkv}")


def test_bulk_wait_timeout_reports_status_and_context_survives():
    # The bulk schedule is told never to issue its copies: its bounded waits
    # run out (2 ms), the status word records it, and the context stays usable.
    binding.device_status(clear=True)
    qkv, wq, wk, pos = qkv_inputs(4, 4, 2, 128, positions="arange", seed=9)
    table = torch.from_numpy(oracle_table(1e6, 8, 128)).cuda()
    q = qkv.cuda()
    binding.qk_norm_rope_fwd(q, wq.cuda(), wk.cuda(), table, pos.cuda(), 4, 2, 128, 128, 1e-6,
                             schedule=binding.RN_QK_BULK, wait_timeout_ns=2_000_000,
                             debug_flags=1)
    assert binding.device_status(clear=True) & binding.RN_STATUS_WAIT_TIMEOUT
    got, want = run_case(4, 4, 2, 128, 128, positions="arange", schedule=binding.RN_QK_BULK,
                         seed=9)
    assert_parity(got, want, "after timeout")
    assert binding.device_status(clear=True) == 0


@pytest.mark.parametrize("T", [1, 2, 16, 64, 256])
def test_small_token_counts_full_rotary(T):
    # packed QKV [T, 48*128], 32 query + 8 key heads, rotary 128, theta 1e6,
    # positions 0..T-1, eps 1e-6
    got, want = run_case(T, 32, 8, 128, 128, positions="arange", max_pos=T)
    assert_parity(got, want, f"T={T}")


@pytest.mark.parametrize("r", [128, 64])
@pytest.mark.parametrize("T", [1024, 4096, 16384])
def test_large_token_counts_full_compare(T, r):
    # positions uniform in [0, 131072); norm over all 128, rotary on the first r
    got, want = run_case(T, 32, 8, 128, r, positions="uniform", max_pos=131072,
                         device_inputs=True, seed=0)
    assert_parity(got, want, f"T={T} r={r}")


def test_schedules_agree_at_scale():
    a, want = run_case(4096, 32, 8, 128, 64, positions="uniform", max_pos=131072,
                       schedule=binding.RN_QK_FOUR_HEADS, device_inputs=True)
    b, _ = run_case(4096, 32, 8, 128, 64, positions="uniform", max_pos=131072,
                    schedule=binding.RN_QK_PERSISTENT, device_inputs=True)
    assert_parity(a, want, "four heads")
    assert np.array_equal(a, b)  # same lane layout and arithmetic: bit-identical


@pytest.mark.parametrize("D,r,style,bf16_table,twin", [
    (128, 64, binding.RN_ROPE_NEOX, False, binding.RN_QK_BULK),
    (128, 128, binding.RN_ROPE_NEOX, False, binding.RN_QK_BULK),
    (128, 32, binding.RN_ROPE_NEOX, False, binding.RN_QK_BULK),
    (128, 128, binding.RN_ROPE_GPTJ, False, binding.RN_QK_FOUR_HEADS),
    (128, 64, binding.RN_ROPE_NEOX, True, binding.RN_QK_FOUR_HEADS),
    (128, 32, binding.RN_ROPE_GPTJ, True, binding.RN_QK_FOUR_HEADS),
])
def test_pairs_bit_identical_to_their_twin(D, r, style, bf16_table, twin):
    # At D 128 the pairs share the 8-lane layout of the ring and of the
    # four-heads kernel, and take the ring's packed arithmetic for neox with an
    # fp32 table and the four-heads kernel's scalar arithmetic otherwise:
    # bit-identical to that schedule.
    Hq, Hkv = 32, 8
    a, want = run_case(3001, Hq, Hkv, D, r, positions="uniform", max_pos=131072,
                       schedule=binding.RN_QK_PAIRS, device_inputs=True, seed=D + r,
                       style=style, bf16_table=bf16_table)
    b, _ = run_case(3001, Hq, Hkv, D, r, positions="uniform", max_pos=131072, schedule=twin,
                    device_inputs=True, seed=D + r, style=style, bf16_table=bf16_table)
    assert_parity(a, want, f"pairs D={D} r={r} style={style} bf16 table={bf16_table}")
    assert np.array_equal(a, b)


@pytest.mark.parametrize("T", [9, 3000])
def test_checked_positions_skip_bad_tokens(T):
    Hq, Hkv, D, r = 4, 2, 128, 128
    max_pos = 64
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions="uniform", max_pos=max_pos, seed=11)
    bad = [1, 4, 8] + ([1500, 2999] if T > 9 else [])
    pos[1] = -1
    pos[4] = max_pos
    pos[8] = max_pos + 1000
    if T > 9:
        pos[1500] = -(1 << 40)
        pos[2999] = 1 << 40
    table = oracle_table(1e6, max_pos, r)
    good_pos = pos.clone()
    good_pos[bad] = 0
    want = oracle.qk_norm_rope(bf16_bits(qkv), bf16_bits(wq), bf16_bits(wk), table,
                               good_pos.numpy(), Hq, Hkv, D, r, 1e-6)
    q = qkv.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.qk_norm_rope_fwd_checked(q, wq.cuda(), wk.cuda(), torch.from_numpy(table).cuda(),
                                     pos.cuda(), Hq, Hkv, D, r, 1e-6, err)
    got = bf16_bits(q).reshape(T, -1)
    assert int(err.item()) & binding.RN_STATUS_BAD_POSITION
    src = bf16_bits(qkv).reshape(T, -1)
    ok_rows = [t for t in range(T) if t not in bad]
    assert np.array_equal(got[bad], src[bad])
    assert_parity(got[ok_rows], want.reshape(T, -1)[ok_rows], "checked good tokens")
    # all positions valid: no flag
    err.zero_()
    q2 = qkv.cuda()
    binding.qk_norm_rope_fwd_checked(q2, wq.cuda(), wk.cuda(), torch.from_numpy(table).cuda(),
                                     good_pos.cuda(), Hq, Hkv, D, r, 1e-6, err)
    assert int(err.item()) == 0


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (32, 8)])
def test_pairs_checked_positions(Hq, Hkv):
    # The pairs schedule checks the second head's position on its own when it
    # belongs to another token: with 6 heads a token a group often holds one
    # head of a rejected token and one of an accepted one.
    T, D, r, max_pos = 3000, 128, 128, 64
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions="uniform", max_pos=max_pos, seed=41)
    bad = [0, 1, 3, 700, 701, 2998]
    for i, t in enumerate(bad):
        pos[t] = -1 - i if i % 2 else max_pos + i
    table = oracle_table(1e6, max_pos, r)
    good_pos = pos.clone()
    good_pos[bad] = 0
    want = oracle.qk_norm_rope(bf16_bits(qkv), bf16_bits(wq), bf16_bits(wk), table,
                               good_pos.numpy(), Hq, Hkv, D, r, 1e-6).reshape(T, -1)
    q = qkv.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.qk_norm_rope_fwd_ex(q, wq.cuda(), wk.cuda(), torch.from_numpy(table).cuda(),
                                pos.cuda(), Hq, Hkv, D, r, 1e-6, max_pos=max_pos, err_flag=err,
                                schedule=binding.RN_QK_PAIRS)
    got = bf16_bits(q).reshape(T, -1)
    assert int(err.item()) & binding.RN_STATUS_BAD_POSITION
    assert np.array_equal(got[bad], bf16_bits(qkv).reshape(T, -1)[bad]), "rejected tokens touched"
    ok_rows = [t for t in range(T) if t not in bad]
    assert_parity(got[ok_rows], want[ok_rows], f"pairs checked Hq={Hq} Hkv={Hkv}")


def test_empty_tokens_is_noop():
    q = torch.empty(0, 48 * 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(4, 128, dtype=torch.float32, device="cuda")
    p = torch.empty(0, dtype=torch.int64, device="cuda")
    binding.qk_norm_rope_fwd(q, w, w, t, p, 32, 8, 128, 128, 1e-6)


@pytest.mark.parametrize("theta,max_pos,r", [(1e6, 131072, 128), (1e6, 131072, 64),
                                             (10000.0, 4096, 64), (500000.0, 333, 32)])
def test_table_builder_matches_oracle(theta, max_pos, r):
    ref = oracle_table(theta, max_pos, r).astype(np.float64)
    got = binding.rope_cos_sin_table(theta, max_pos, r).cpu().numpy().astype(np.float64)
    # Both sides evaluate in double and round once to float; pow/sin/cos may
    # differ in the last double bit, which at angles up to 1.3e5 rad moves the
    # value by ~3e-11: allow one float step plus that.
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= ulp + 1e-10)
    assert np.mean(got == ref) > 0.999


@pytest.mark.parametrize("schedule", [binding.RN_QK_FOUR_HEADS, binding.RN_QK_BULK,
                                      binding.RN_QK_PAIRS])
def test_positions_view_at_8_byte_offset(schedule):
    # positions only need 8-byte alignment: a view one int64 into a buffer works
    T, Hq, Hkv, D, r = 2049, 4, 2, 128, 64
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions="uniform", max_pos=500, seed=21)
    table = oracle_table(1e6, 500, r)
    want = oracle.qk_norm_rope(bf16_bits(qkv[1:]), bf16_bits(wq), bf16_bits(wk), table,
                               pos[1:].numpy(), Hq, Hkv, D, r, 1e-6)
    q = qkv[1:].cuda()
    pos_view = pos.cuda()[1:]
    assert pos_view.data_ptr() % 16 == 8
    binding.qk_norm_rope_fwd(q, wq.cuda(), wk.cuda(), torch.from_numpy(table).cuda(), pos_view,
                             Hq, Hkv, D, r, 1e-6, schedule=schedule)
    assert_parity(bf16_bits(q), want, f"offset positions sched={schedule}")


# ---------------------------------------------------------------------------
# GPT-J (interleaved) rotary pairing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("schedule", QK_SCHEDULES)
@pytest.mark.parametrize("D,r", LAYOUTS)
def test_gptj_layouts_every_schedule(D, r, schedule):
    if schedule in NOT_64_16 and (D, r) == (64, 16):
        return  # the ring does not take this layout (the warp schedules do)
    got, want = run_case(5, 4, 2, D, r, positions="uniform", max_pos=97, schedule=schedule,
                         seed=D + r + 1, style=binding.RN_ROPE_GPTJ)
    assert_parity(got, want, f"gptj D={D} r={r} sched={schedule}")


@pytest.mark.parametrize("schedule", [binding.RN_QK_AUTO, binding.RN_QK_FOUR_HEADS,
                                      binding.RN_QK_BULK, binding.RN_QK_PAIRS])
@pytest.mark.parametrize("r", [128, 64])
def test_gptj_many_tokens_full_compare(r, schedule):
    got, want = run_case(4096, 32, 8, 128, r, positions="uniform", max_pos=131072,
                         device_inputs=True, seed=3, schedule=schedule,
                         style=binding.RN_ROPE_GPTJ)
    assert_parity(got, want, f"gptj T=4096 r={r} sched={schedule}")


def test_gptj_checked_positions():
    T, Hq, Hkv, D, r = 3000, 4, 2, 128, 64
    max_pos = 64
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions="uniform", max_pos=max_pos, seed=12)
    pos[5] = -3
    pos[2222] = max_pos
    table = oracle_table(1e6, max_pos, r)
    good = pos.clone()
    good[[5, 2222]] = 0
    want = oracle.qk_norm_rope(bf16_bits(qkv), bf16_bits(wq), bf16_bits(wk), table,
                               good.numpy(), Hq, Hkv, D, r, 1e-6, style=1).reshape(T, -1)
    q = qkv.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.qk_norm_rope_fwd_ex(q, wq.cuda(), wk.cuda(), torch.from_numpy(table).cuda(),
                                pos.cuda(), Hq, Hkv, D, r, 1e-6, rope_style=binding.RN_ROPE_GPTJ,
                                max_pos=max_pos, err_flag=err)
    got = bf16_bits(q).reshape(T, -1)
    assert int(err.item()) & binding.RN_STATUS_BAD_POSITION
    src = bf16_bits(qkv).reshape(T, -1)
    assert np.array_equal(got[[5, 2222]], src[[5, 2222]])
    ok_rows = [t for t in range(T) if t not in (5, 2222)]
    assert_parity(got[ok_rows], want[ok_rows], "gptj checked")


# ---------------------------------------------------------------------------
# bf16 cos/sin table
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("style", [binding.RN_ROPE_NEOX, binding.RN_ROPE_GPTJ])
@pytest.mark.parametrize("schedule", QK_SCHEDULES)
@pytest.mark.parametrize("D,r", LAYOUTS)
def test_bf16_table_layouts_every_schedule(D, r, schedule, style):
    if schedule in NOT_64_16 and (D, r) == (64, 16):
        return  # the ring does not take this layout (the warp schedules do)
    got, want = run_case(7, 4, 2, D, r, positions="uniform", max_pos=211, schedule=schedule,
                         seed=D + 3 * r + style, style=style, bf16_table=True)
    assert_parity(got, want, f"bf16 table D={D} r={r} sched={schedule} style={style}")


@pytest.mark.parametrize("style", [binding.RN_ROPE_NEOX, binding.RN_ROPE_GPTJ])
@pytest.mark.parametrize("schedule", [binding.RN_QK_AUTO, binding.RN_QK_PERSISTENT,
                                      binding.RN_QK_BULK, binding.RN_QK_PAIRS])
@pytest.mark.parametrize("r", [128, 64])
def test_bf16_table_many_tokens_full_compare(r, schedule, style):
    # 16384 tokens (4096 for the warp grids), uniform positions over 131072
    T = 4096 if schedule in (binding.RN_QK_PERSISTENT, binding.RN_QK_PAIRS) else 16384
    got, want = run_case(T, 32, 8, 128, r, positions="uniform", max_pos=131072,
                         device_inputs=True, seed=17 + r, schedule=schedule, style=style,
                         bf16_table=True)
    assert_parity(got, want, f"bf16 table T={T} r={r} sched={schedule} style={style}")


def test_bf16_table_checked_positions():
    T, Hq, Hkv, D, r = 3000, 4, 2, 128, 128
    max_pos = 64
    qkv, wq, wk, pos = qkv_inputs(T, Hq, Hkv, D, positions="uniform", max_pos=max_pos, seed=31)
    bad = torch.arange(0, T, 7)
    pos[bad] = torch.where(bad % 2 == 0, torch.tensor(-1), torch.tensor(max_pos + 5))
    dev_table, table = oracle_table_bf16(1e6, max_pos, r)
    good = (pos >= 0) & (pos < max_pos)
    want = bf16_bits(qkv).copy()
    ok_rows = good.numpy()
    want[ok_rows] = oracle.qk_norm_rope(bf16_bits(qkv[good]), bf16_bits(wq), bf16_bits(wk), table,
                                        pos[good].numpy(), Hq, Hkv, D, r, 1e-6)
    for schedule in (binding.RN_QK_FOUR_HEADS, binding.RN_QK_BULK, binding.RN_QK_PAIRS):
        q = qkv.cuda()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.qk_norm_rope_fwd_ex(q, wq.cuda(), wk.cuda(), dev_table, pos.cuda(), Hq, Hkv, D, r,
                                    1e-6, max_pos=max_pos, err_flag=err, schedule=schedule)
        assert int(err.item()) & binding.RN_STATUS_BAD_POSITION
        got = bf16_bits(q)
        assert np.array_equal(got[~ok_rows], bf16_bits(qkv)[~ok_rows]), "rejected tokens touched"
        assert_parity(got[ok_rows], want[ok_rows], f"bf16 table checked sched={schedule}")


@pytest.mark.parametrize("theta,max_pos,r", [(1e6, 131072, 128), (1e6, 131072, 64),
                                             (10000.0, 4096, 64), (500000.0, 333, 32)])
def test_bf16_table_builder_matches_oracle(theta, max_pos, r):
    ref = oracle.rope_cos_sin_bf16(theta, max_pos, r)
    got = bf16_bits(binding.rope_cos_sin_table(theta, max_pos, r, dtype=torch.bfloat16))
    # Both sides round the double value once to bf16; pow/sin/cos may differ
    # in the last double bit, which flips the rounding only for a value within
    # ~1e-10 of a bf16 midpoint: at most a step, and almost never.
    from tests.exact import ulp_distance_bf16
    d = ulp_distance_bf16(got, ref)
    assert d.max() <= 1
    assert np.mean(d == 0) > 0.99999


@pytest.mark.parametrize("r", [128, 64])
def test_device_and_host_tables_agree(r):
    # rope_cos_sin_table (fp64 on the device) and rope_cos_sin_table_host (fp64
    # on the CPU) round their angles once to fp32.  The two fp64 pow and
    # sincos may differ in the last bit: f_i by a few 2^-53 relative, so the
    # angle p * f_i by under 1e-10 for p < 2^17.  An entry then differs by one
    # fp32 step at most, or, where cos or sin is near zero and a step is
    # tiny, by at most 1e-10 absolute.
    dev = binding.rope_cos_sin_table(1e6, 131072, r).cpu().numpy()
    host = binding.rope_cos_sin_table(1e6, 131072, r, device="cpu").numpy()
    steps = np.abs(dev.view(np.int32).astype(np.int64) - host.view(np.int32).astype(np.int64))
    close = np.abs(dev.astype(np.float64) - host.astype(np.float64)) <= 1e-10
    assert np.all((steps <= 1) | close)
    assert np.count_nonzero(steps) <= dev.size * 1e-3
