"""The C-ABI library loads and exports every symbol row_norm.h declares, and
its host-side argument checks answer before anything touches a device
(CPU only: no compute call is made here)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from row_normalization_gb300 import binding
from row_normalization_gb300.build import ROOT, build

HEADER = os.path.join(ROOT, "include", "row_norm.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("rmsnorm_fwd", "add_rmsnorm_fwd", "qk_norm_rope_fwd", "qk_norm_rope_fwd_checked",
                     "rope_cos_sin_table", "rn_error_string", "rn_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in row_norm.h but not exported"


def test_error_strings_and_version(lib):
    assert binding.error_string(0) == "ok"
    for code in range(-6, 0):
        s = binding.error_string(code)
        assert s and s != "unknown status code"
    assert binding.error_string(-99) == "unknown status code"
    assert binding.version() >= 100


# Fake but well-formed pointer values: the checks below must reject the call
# before any of them is dereferenced or handed to the driver.
P = 0x10000
MISALIGNED = 0x10008


@pytest.mark.parametrize("M,N,expect", [
    (4, 7, binding.RN_ERR_SHAPE),       # N % 8 != 0
    (4, 0, binding.RN_ERR_SHAPE),
    (4, 65544, binding.RN_ERR_SHAPE),   # N > 65536
    (-1, 64, binding.RN_ERR_SHAPE),
    (0, 64, binding.RN_OK),             # empty: no-op
])
def test_rmsnorm_shape_checks(lib, M, N, expect):
    assert lib.rmsnorm_fwd(P, P, 1e-6, M, N, P, None) == expect


def test_rmsnorm_null_and_alignment_checks(lib):
    assert lib.rmsnorm_fwd(None, P, 1e-6, 4, 64, P, None) == binding.RN_ERR_NULL
    assert lib.rmsnorm_fwd(P, None, 1e-6, 4, 64, P, None) == binding.RN_ERR_NULL
    assert lib.rmsnorm_fwd(P, P, 1e-6, 4, 64, None, None) == binding.RN_ERR_NULL
    assert lib.rmsnorm_fwd(MISALIGNED, P, 1e-6, 4, 64, P, None) == binding.RN_ERR_ALIGN
    assert lib.rmsnorm_fwd(P, P, 1e-6, 4, 64, MISALIGNED, None) == binding.RN_ERR_ALIGN
    assert lib.rmsnorm_fwd_sched(P, P, 1e-6, 4, 64, P, 9, 0, 0, None) == binding.RN_ERR_ARG


@pytest.mark.parametrize("T,Hq,Hkv,D,r,expect", [
    (4, 32, 8, 96, 96, binding.RN_ERR_SHAPE),     # D unsupported
    (4, 32, 8, 128, 127, binding.RN_ERR_SHAPE),   # odd rotary_dim
    (4, 32, 8, 128, 256, binding.RN_ERR_SHAPE),   # rotary_dim > D
    (4, 32, 8, 128, 48, binding.RN_ERR_SHAPE),    # rotary_dim not D, D/2 or D/4
    (-1, 32, 8, 128, 128, binding.RN_ERR_SHAPE),
    (4, -1, 8, 128, 128, binding.RN_ERR_SHAPE),
    (0, 32, 8, 128, 128, binding.RN_OK),          # no tokens
    (4, 0, 0, 128, 128, binding.RN_OK),           # no Q/K heads
    (1 << 26, 32, 8, 128, 128, binding.RN_ERR_SHAPE),  # T*(Hq+Hkv) >= 2^31
])
def test_qk_shape_checks(lib, T, Hq, Hkv, D, r, expect):
    assert lib.qk_norm_rope_fwd(P, P, P, P, P, T, Hq, Hkv, D, r, 1e-6, None) == expect


def test_qk_null_alignment_and_checked_args(lib):
    assert lib.qk_norm_rope_fwd(P, P, None, P, P, 4, 2, 1, 128, 128, 1e-6, None) == binding.RN_ERR_NULL
    assert lib.qk_norm_rope_fwd(P, P, P, P, P + 4, 4, 2, 1, 128, 128, 1e-6, None) == binding.RN_ERR_ALIGN
    assert lib.qk_norm_rope_fwd(P, P, P, MISALIGNED, P, 4, 2, 1, 128, 128, 1e-6, None) == binding.RN_ERR_ALIGN
    assert lib.qk_norm_rope_fwd_checked(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 0, P, None) == binding.RN_ERR_SHAPE
    assert lib.qk_norm_rope_fwd_checked(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 16, None, None) == binding.RN_ERR_NULL
    assert lib.qk_norm_rope_fwd_sched(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 3, 0, 0, None) == binding.RN_ERR_ARG


def test_add_rmsnorm_checks(lib):
    assert lib.add_rmsnorm_fwd(P, P, P, 1e-6, 4, 7, P, P + 4096, None) == binding.RN_ERR_SHAPE
    assert lib.add_rmsnorm_fwd(P, P, P, 1e-6, 0, 64, P, P + 4096, None) == binding.RN_OK
    assert lib.add_rmsnorm_fwd(P, None, P, 1e-6, 4, 64, P, P + 4096, None) == binding.RN_ERR_NULL
    assert lib.add_rmsnorm_fwd(P, P, P, 1e-6, 4, 64, MISALIGNED, P + 4096, None) == binding.RN_ERR_ALIGN
    assert lib.add_rmsnorm_fwd(P, P, P, 1e-6, 4, 64, P + 4096, P + 4096, None) == binding.RN_ERR_ARG


def test_l2norm_checks(lib):
    assert lib.l2norm_fwd(P, 1e-12, 4, 7, P, None) == binding.RN_ERR_SHAPE
    assert lib.l2norm_fwd(P, 1e-12, 0, 64, P, None) == binding.RN_OK
    assert lib.l2norm_fwd(None, 1e-12, 4, 64, P, None) == binding.RN_ERR_NULL
    assert lib.l2norm_fwd(P, 1e-12, 4, 64, MISALIGNED, None) == binding.RN_ERR_ALIGN


def test_layernorm_checks(lib):
    assert lib.layernorm_fwd(P, P, None, 1e-5, 4, 7, P, None) == binding.RN_ERR_SHAPE
    assert lib.layernorm_fwd(P, P, None, 1e-5, 0, 64, P, None) == binding.RN_OK
    assert lib.layernorm_fwd(P, None, P, 1e-5, 4, 64, P, None) == binding.RN_ERR_NULL
    assert lib.layernorm_fwd(P, P, MISALIGNED, 1e-5, 4, 64, P, None) == binding.RN_ERR_ALIGN
    assert lib.layernorm_fwd_sched(P, P, None, 1e-5, 4, 64, P, 7, 0, 0, None) == binding.RN_ERR_ARG


def test_qk_ex_checks(lib):
    # unknown rope style, negative max_pos, checked mode without a flag pointer
    assert lib.qk_norm_rope_fwd_ex(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 2, 0, None, 0, 0, 0, None) == binding.RN_ERR_ARG
    assert lib.qk_norm_rope_fwd_ex(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 1, -1, None, 0, 0, 0, None) == binding.RN_ERR_SHAPE
    assert lib.qk_norm_rope_fwd_ex(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 1, 16, None, 0, 0, 0, None) == binding.RN_ERR_NULL


def test_qk_ex_bf16_table_checks(lib):
    f = lib.qk_norm_rope_fwd_ex_bf16_table
    assert f(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 2, 0, None, 0, 0, 0, None) == binding.RN_ERR_ARG
    assert f(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 1, -1, None, 0, 0, 0, None) == binding.RN_ERR_SHAPE
    assert f(P, P, P, P, P, 4, 2, 1, 128, 128, 1e-6, 1, 16, None, 0, 0, 0, None) == binding.RN_ERR_NULL
    assert f(P, P, P, MISALIGNED, P, 4, 2, 1, 128, 128, 1e-6, 0, 0, None, 0, 0, 0, None) == binding.RN_ERR_ALIGN
    assert f(P, P, P, None, P, 4, 2, 1, 128, 128, 1e-6, 0, 0, None, 0, 0, 0, None) == binding.RN_ERR_NULL
    assert f(P, P, P, P, P, 4, 2, 1, 128, 96, 1e-6, 0, 0, None, 0, 0, 0, None) == binding.RN_ERR_SHAPE
    assert f(P, P, P, P, P, 0, 2, 1, 128, 128, 1e-6, 0, 0, None, 0, 0, 0, None) == binding.RN_OK


@pytest.mark.parametrize("fn", ["rope_cos_sin_table", "rope_cos_sin_table_bf16"])
def test_table_checks(lib, fn):
    f = getattr(lib, fn)
    assert f(1e6, 16, 7, P, None) == binding.RN_ERR_SHAPE
    assert f(-1.0, 16, 8, P, None) == binding.RN_ERR_SHAPE
    assert f(1e6, 0, 8, P, None) == binding.RN_OK
    assert f(1e6, 16, 8, None, None) == binding.RN_ERR_NULL
    assert f(1e6, 16, 8, MISALIGNED, None) == binding.RN_ERR_ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_no_device_is_reported_not_crashed(lib):
    # Well-formed arguments on a host without a GPU: the library must answer
    # RN_ERR_DEVICE instead of launching.
    assert lib.rmsnorm_fwd(P, P, 1e-6, 4, 64, P, None) == binding.RN_ERR_DEVICE
    v = ctypes.c_uint(0)
    assert lib.rn_device_status(ctypes.byref(v), 0) == binding.RN_ERR_DEVICE


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    import row_normalization_gb300.binding as b
    saved = b._lib
    try:
        b._lib = None
        with pytest.raises(RuntimeError, match="build the CUDA library"):
            b.load(str(tmp_path / "missing.so"))
    finally:
        b._lib = saved
        importlib.invalidate_caches()


# ---- fp16 row norms and the general row entry point -----------------------

@pytest.mark.parametrize("M,N,expect", [
    (4, 7, binding.RN_ERR_SHAPE), (4, 65544, binding.RN_ERR_SHAPE), (-1, 64, binding.RN_ERR_SHAPE),
    (0, 64, binding.RN_OK),
])
def test_f16_entry_points_shape_checks(lib, M, N, expect):
    assert lib.rmsnorm_fwd_f16(P, P, 1e-6, M, N, P, None) == expect
    assert lib.l2norm_fwd_f16(P, 1e-6, M, N, P, None) == expect
    assert lib.add_rmsnorm_fwd_f16(P, P, P, 1e-6, M, N, P, P + 4096, None) == expect
    assert lib.layernorm_fwd_f16(P, P, None, 1e-6, M, N, P, None) == expect


def test_f16_entry_points_null_alignment_and_aliasing(lib):
    assert lib.rmsnorm_fwd_f16(None, P, 1e-6, 4, 64, P, None) == binding.RN_ERR_NULL
    assert lib.rmsnorm_fwd_f16(P, P, 1e-6, 4, 64, MISALIGNED, None) == binding.RN_ERR_ALIGN
    assert lib.l2norm_fwd_f16(MISALIGNED, 1e-6, 4, 64, P, None) == binding.RN_ERR_ALIGN
    assert lib.add_rmsnorm_fwd_f16(P, None, P, 1e-6, 4, 64, P, P, None) == binding.RN_ERR_NULL
    assert lib.add_rmsnorm_fwd_f16(P, P, P, 1e-6, 4, 64, P, P, None) == binding.RN_ERR_ARG
    assert lib.layernorm_fwd_f16(P, P, MISALIGNED, 1e-6, 4, 64, P, None) == binding.RN_ERR_ALIGN


def test_row_norm_fwd_ex_checks(lib):
    ex = lib.row_norm_fwd_ex
    # unknown op or element format
    assert ex(4, 0, P, None, P, None, 1e-6, 4, 64, None, P, 0, 0, 0, None) == binding.RN_ERR_ARG
    assert ex(-1, 0, P, None, P, None, 1e-6, 4, 64, None, P, 0, 0, 0, None) == binding.RN_ERR_ARG
    assert ex(0, 2, P, None, P, None, 1e-6, 4, 64, None, P, 0, 0, 0, None) == binding.RN_ERR_ARG
    for dt in (binding.RN_DTYPE_BF16, binding.RN_DTYPE_F16):
        # pointers an op does not use are ignored: a misaligned residual, h and
        # bias pass the checks of plain RMSNorm, which then stops at the bad
        # schedule (checked after the pointers)
        assert ex(binding.RN_OP_RMSNORM, dt, P, MISALIGNED, P, MISALIGNED, 1e-6, 4, 64,
                  MISALIGNED, P, 9, 0, 0, None) == binding.RN_ERR_ARG
        # L2Norm takes no weight
        assert ex(binding.RN_OP_L2NORM, dt, P, None, None, None, 1e-6, 4, 64, None, P, 9, 0, 0,
                  None) == binding.RN_ERR_ARG
        # the fused add needs its residual and h, distinct from y
        assert ex(binding.RN_OP_ADD_RMSNORM, dt, P, None, P, None, 1e-6, 4, 64, P + 4096, P, 0,
                  0, 0, None) == binding.RN_ERR_NULL
        assert ex(binding.RN_OP_ADD_RMSNORM, dt, P, P, P, None, 1e-6, 4, 64, P, P, 0, 0, 0,
                  None) == binding.RN_ERR_ARG
        assert ex(binding.RN_OP_LAYERNORM, dt, P, None, P, MISALIGNED, 1e-6, 4, 64, None, P, 0,
                  0, 0, None) == binding.RN_ERR_ALIGN
        assert ex(binding.RN_OP_LAYERNORM, dt, P, None, P, None, 1e-6, 0, 64, None, P, 0, 0, 0,
                  None) == binding.RN_OK
    assert lib.row_norm_select_schedule(7, 8, 64) == binding.RN_ERR_ARG
    assert lib.row_norm_select_schedule(0, 8, 7) == binding.RN_ERR_SHAPE


def test_binding_rejects_mixed_and_unsupported_dtypes():
    x = torch.zeros(2, 8, dtype=torch.float32)
    with pytest.raises(TypeError):
        binding.rmsnorm_fwd(x, torch.zeros(8), 1e-6)
    with pytest.raises((TypeError, ValueError)):
        binding.rmsnorm_fwd(torch.zeros(2, 8, dtype=torch.float16),
                            torch.zeros(8, dtype=torch.bfloat16), 1e-6)


def test_workspace_forms_checks(lib):
    # the header's workspace size is the binding's
    text = open(HEADER).read()
    assert int(re.search(r"#define RN_WORKSPACE_BYTES (\d+)", text).group(1)) == \
        binding.RN_WORKSPACE_BYTES
    # a misaligned workspace is refused before anything is launched
    assert lib.rmsnorm_fwd_ws(P, P, 1e-6, 4, 64, P, MISALIGNED, None) == binding.RN_ERR_ALIGN
    assert lib.rmsnorm_fwd_ws(P, P, 1e-6, 4, 7, P, P, None) == binding.RN_ERR_SHAPE
    assert lib.rmsnorm_fwd_ws(P, P, 1e-6, 0, 64, P, P, None) == binding.RN_OK
    assert lib.row_norm_fwd_ws(9, 0, P, P, P, P, 1e-6, 4, 64, P, P, P, 0, 0, 0, None) == binding.RN_ERR_ARG
    assert lib.row_norm_fwd_ws(0, 0, P, None, P, None, 1e-6, 4, 64, None, P, MISALIGNED, 0, 0, 0,
                               None) == binding.RN_ERR_ALIGN


def test_header_constants_are_the_bindings():
    # every enum value and #define the header gives a caller is in the binding,
    # with the same value
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    consts = {n: int(v) for n, v in re.findall(r"\b(RN_[A-Z0-9_]+)\s*=\s*(-?\d+)u?\b", text)}
    consts.update({n: int(v) for n, v in re.findall(r"#define\s+(RN_[A-Z0-9_]+)\s+(\d+)\b", text)})
    assert {"RN_QK_PAIRS", "RN_SCHED_PERSIST_BULK", "RN_ERR_ARG", "RN_OP_LAYERNORM"} <= set(consts)
    for name, value in consts.items():
        assert getattr(binding, name) == value, name


def test_qk_schedule_selection_by_layout(lib):
    # host-only: the automatic pick by token count and layout, at its boundaries
    sel = binding.qk_norm_rope_select_schedule
    assert [sel(T) for T in (1, 2, 3, 256, 257, 1023, 1024, 5120, 5121)] == [
        binding.RN_QK_HEAD_PER_WARP, binding.RN_QK_HEAD_PER_WARP, binding.RN_QK_TWO_HEADS,
        binding.RN_QK_TWO_HEADS, binding.RN_QK_PERSISTENT, binding.RN_QK_PERSISTENT,
        binding.RN_QK_PAIRS, binding.RN_QK_PAIRS, binding.RN_QK_BULK]
    assert sel(4096, 128, 64) == binding.RN_QK_PAIRS and sel(4097, 128, 64) == binding.RN_QK_BULK
    assert sel(6144, 256, 128) == binding.RN_QK_PAIRS and sel(6145, 256, 128) == binding.RN_QK_BULK
    assert sel(1023, 128, 64) == binding.RN_QK_PERSISTENT and sel(1024, 128, 64) == binding.RN_QK_PAIRS
    assert sel(1791, 128, 32) == binding.RN_QK_PERSISTENT and sel(1792, 128, 32) == binding.RN_QK_PAIRS
    assert lib.qk_norm_rope_select_schedule(3000) == sel(3000, 128, 128)
    for r in (128, 64, 32):
        assert sel(1 << 20, 128, r) == binding.RN_QK_BULK
    # the ring never: 64-wide heads and 256-wide with full rotary take the pairs
    for D, r in ((64, 64), (64, 32), (64, 16), (256, 256)):
        assert sel(1 << 20, D, r) == binding.RN_QK_PAIRS
    assert sel(1023, 64, 64) == binding.RN_QK_PERSISTENT and sel(1024, 64, 64) == binding.RN_QK_PAIRS
    assert sel(3071, 64, 16) == binding.RN_QK_PERSISTENT and sel(3072, 64, 16) == binding.RN_QK_PAIRS
    assert sel(257, 256, 256) == binding.RN_QK_PAIRS and sel(257, 256, 128) == binding.RN_QK_PAIRS
    assert sel(1 << 20, 256, 128) == binding.RN_QK_BULK
    # rotary 64 of 256: the pairs from 512 through 4096 tokens, the four-heads grid around them
    assert [sel(T, 256, 64) for T in (511, 512, 4096, 4097, 1 << 20)] == [
        binding.RN_QK_PERSISTENT, binding.RN_QK_PAIRS, binding.RN_QK_PAIRS,
        binding.RN_QK_PERSISTENT, binding.RN_QK_PERSISTENT]
    for T, D, r in ((-1, 128, 128), (100, 96, 96), (100, 128, 48), (100, 128, 16)):
        assert lib.qk_norm_rope_select_schedule_ex(T, D, r) == binding.RN_ERR_SHAPE
    with pytest.raises(binding.RowNormError):
        sel(100, 128, 48)
