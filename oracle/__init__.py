"""fp64 CPU oracle for bf16 row normalization -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library never calls it
and shares no code with it.

The arithmetic lives in ``rn_oracle.c`` (plain C, double precision, one
bf16 rounding at the end).  This module compiles it with gcc on first use
(or through :func:`build`) and exposes numpy-level wrappers.  Inputs and
outputs are raw bf16 bit patterns held in ``numpy.uint16`` arrays.

Passages followed:
  * RMSNorm -- "[Inductor] Codegen Gluon", section 3.1.
  * fused Q/K RMSNorm + neox RoPE -- "[pretuned] Optimize fused_qk_norm_rope
    on B200", section "Summary".
  * L2Norm -- "[Inductor] Codegen Gluon", section 3.2.
  * fused residual add + RMSNorm -- "TorchInductor: from ATen IR to Triton
    kernel", sections 14.3 and 14.27.
  * LayerNorm -- "TorchInductor: from ATen IR to Triton kernel", section
    14.12.2.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "librn_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``rn_oracle.c`` into a shared library with gcc and return its path.

    ``-ffp-contract=off`` keeps a*b+c as two rounded operations on every host
    (gcc on aarch64 would otherwise fuse them), so x86 and Arm agree bit for
    bit.  No fast-math.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # A test may point this at a deliberately broken build of the oracle
        # to show that the pins catch it.
        override = os.environ.get("RN_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.rn_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.rn_oracle_bf16_to_double.restype = ctypes.c_double
        lib.rn_oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.rn_oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.rn_oracle_rmsnorm.argtypes = [u16p, u16p, ctypes.c_float,
                                          ctypes.c_int64, ctypes.c_int64, u16p]
        lib.rn_oracle_rmsnorm.restype = ctypes.c_int
        lib.rn_oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.rn_oracle_f16_to_double.restype = ctypes.c_double
        lib.rn_oracle_double_to_f16.argtypes = [ctypes.c_double]
        lib.rn_oracle_double_to_f16.restype = ctypes.c_uint16
        i32 = ctypes.c_int
        lib.rn_oracle_rmsnorm_fmt.argtypes = lib.rn_oracle_rmsnorm.argtypes + [i32]
        lib.rn_oracle_rmsnorm_fmt.restype = i32
        lib.rn_oracle_l2norm_fmt.argtypes = [u16p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                             u16p, i32]
        lib.rn_oracle_l2norm_fmt.restype = i32
        lib.rn_oracle_add_rmsnorm_fmt.argtypes = [u16p, u16p, u16p, ctypes.c_float, ctypes.c_int64,
                                                  ctypes.c_int64, u16p, u16p, i32]
        lib.rn_oracle_add_rmsnorm_fmt.restype = i32
        lib.rn_oracle_layernorm_fmt.argtypes = [u16p, u16p, u16p, ctypes.c_float, ctypes.c_int64,
                                                ctypes.c_int64, u16p, i32]
        lib.rn_oracle_layernorm_fmt.restype = i32
        lib.rn_oracle_rms_rstd.argtypes = [u16p, ctypes.c_float, ctypes.c_int64,
                                           ctypes.c_int64, f64p]
        lib.rn_oracle_rms_rstd.restype = ctypes.c_int
        lib.rn_oracle_rope_cos_sin.argtypes = [ctypes.c_double, ctypes.c_int64,
                                               ctypes.c_int, f32p]
        lib.rn_oracle_rope_cos_sin.restype = ctypes.c_int
        lib.rn_oracle_rope_cos_sin_bf16.argtypes = [ctypes.c_double, ctypes.c_int64,
                                                    ctypes.c_int, u16p]
        lib.rn_oracle_rope_cos_sin_bf16.restype = ctypes.c_int
        lib.rn_oracle_qk_norm_rope.argtypes = [
            u16p, u16p, u16p, f32p, i64p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float]
        lib.rn_oracle_qk_norm_rope.restype = ctypes.c_int
        lib.rn_oracle_qk_norm_rope_ex.argtypes = lib.rn_oracle_qk_norm_rope.argtypes + [ctypes.c_int]
        lib.rn_oracle_qk_norm_rope_ex.restype = ctypes.c_int
        lib.rn_oracle_l2norm.argtypes = [u16p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64, u16p]
        lib.rn_oracle_l2norm.restype = ctypes.c_int
        lib.rn_oracle_add_rmsnorm.argtypes = [u16p, u16p, u16p, ctypes.c_float, ctypes.c_int64,
                                              ctypes.c_int64, u16p, u16p]
        lib.rn_oracle_add_rmsnorm.restype = ctypes.c_int
        lib.rn_oracle_layernorm.argtypes = [u16p, u16p, u16p, ctypes.c_float,
                                            ctypes.c_int64, ctypes.c_int64, u16p]
        lib.rn_oracle_layernorm.restype = ctypes.c_int
        _lib = lib
        return lib


class OracleError(ValueError):
    """The oracle rejected its arguments (negative status from the C code)."""


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


# ---- scalar helpers ---------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return float(_load().rn_oracle_bf16_to_double(int(bits) & 0xFFFF))


def double_to_bf16(v: float) -> int:
    """Round one double to the nearest bf16 (ties to even); returns the bits."""
    return int(_load().rn_oracle_double_to_bf16(float(v)))


def f16_to_double(bits: int) -> float:
    return float(_load().rn_oracle_f16_to_double(int(bits) & 0xFFFF))


def double_to_f16(v: float) -> int:
    """Round one double to the nearest IEEE binary16 (ties to even); returns the bits."""
    return int(_load().rn_oracle_double_to_f16(float(v)))


# ---- array entry points -----------------------------------------------------

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float, f16: bool = False) -> np.ndarray:
    """y = round(x * 1/sqrt(mean(x^2) + eps) * w) row by row; x is [M, N] uint16
    bit patterns of bf16 (or IEEE fp16 with f16=True)."""
    x = _u16(x)
    w = _u16(w)
    if x.ndim != 2 or w.shape != (x.shape[1],):
        raise ValueError("x must be [M, N] and w [N]")
    M, N = x.shape
    y = np.zeros_like(x)
    _check(_load().rn_oracle_rmsnorm_fmt(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                                         ctypes.c_float(eps), M, N,
                                         _ptr(y, ctypes.c_uint16), int(f16)), "rmsnorm")
    return y


def rms_rstd(x: np.ndarray, eps: float) -> np.ndarray:
    """Per-row 1/sqrt(mean(x^2) + eps) in float64."""
    x = _u16(x)
    M, N = x.shape
    out = np.zeros(M, dtype=np.float64)
    _check(_load().rn_oracle_rms_rstd(_ptr(x, ctypes.c_uint16), ctypes.c_float(eps),
                                      M, N, _ptr(out, ctypes.c_double)), "rms_rstd")
    return out


def rope_cos_sin(theta: float, max_pos: int, rotary_dim: int) -> np.ndarray:
    """fp32 table [max_pos, rotary_dim]: cos half, then sin half, angle p*theta^(-2i/r)."""
    out = np.zeros((max_pos, rotary_dim), dtype=np.float32)
    _check(_load().rn_oracle_rope_cos_sin(float(theta), int(max_pos), int(rotary_dim),
                                          _ptr(out, ctypes.c_float)), "rope_cos_sin")
    return out


def rope_cos_sin_bf16(theta: float, max_pos: int, rotary_dim: int) -> np.ndarray:
    """bf16 table (uint16 bit patterns) [max_pos, rotary_dim]: the same angles as
    rope_cos_sin, each entry rounded once from double to bf16."""
    out = np.zeros((max_pos, rotary_dim), dtype=np.uint16)
    _check(_load().rn_oracle_rope_cos_sin_bf16(float(theta), int(max_pos), int(rotary_dim),
                                               _ptr(out, ctypes.c_uint16)), "rope_cos_sin_bf16")
    return out


def qk_norm_rope(qkv: np.ndarray, wq: np.ndarray, wk: np.ndarray,
                 cos_sin: np.ndarray, positions: np.ndarray, Hq: int, Hkv: int,
                 D: int, rotary_dim: int, eps: float, style: int = 0) -> np.ndarray:
    """Return a copy of qkv [T, (Hq+2Hkv)*D] with Q/K heads normed and rotated.
    style 0: neox pairs (i, i + r/2); style 1: GPT-J pairs (2i, 2i + 1)."""
    out = _u16(qkv).copy()
    wq = _u16(wq)
    wk = _u16(wk)
    cos_sin = np.ascontiguousarray(cos_sin, dtype=np.float32)
    positions = np.ascontiguousarray(positions, dtype=np.int64)
    T = out.shape[0]
    if out.size != T * (Hq + 2 * Hkv) * D:
        raise ValueError("qkv shape does not match T, Hq, Hkv, D")
    if cos_sin.ndim != 2 or cos_sin.shape[1] != rotary_dim:
        raise ValueError("cos_sin must be [max_pos, rotary_dim]")
    if positions.shape != (T,):
        raise ValueError("positions must be [T]")
    fn = _load().rn_oracle_qk_norm_rope_ex if style else _load().rn_oracle_qk_norm_rope
    extra = (int(style),) if style else ()
    _check(fn(
        _ptr(out, ctypes.c_uint16), _ptr(wq, ctypes.c_uint16), _ptr(wk, ctypes.c_uint16),
        _ptr(cos_sin, ctypes.c_float), _ptr(positions, ctypes.c_int64),
        cos_sin.shape[0], T, Hq, Hkv, D, rotary_dim, ctypes.c_float(eps), *extra), "qk_norm_rope")
    return out


def l2norm(x: np.ndarray, eps: float, f16: bool = False) -> np.ndarray:
    """y = round(x / max(||x||_2, eps)) row by row (bf16, or fp16 with f16=True)."""
    x = _u16(x)
    M, N = x.shape
    y = np.zeros_like(x)
    _check(_load().rn_oracle_l2norm_fmt(_ptr(x, ctypes.c_uint16), ctypes.c_float(eps), M, N,
                                        _ptr(y, ctypes.c_uint16), int(f16)), "l2norm")
    return y


def add_rmsnorm(x: np.ndarray, res: np.ndarray, w: np.ndarray, eps: float, f16: bool = False):
    """(h, y): h = round(x + res), y = rmsnorm(h) row by row (bf16, or fp16)."""
    x = _u16(x)
    res = _u16(res)
    w = _u16(w)
    if x.shape != res.shape or x.ndim != 2 or w.shape != (x.shape[1],):
        raise ValueError("x and res must be [M, N] and w [N]")
    M, N = x.shape
    h = np.zeros_like(x)
    y = np.zeros_like(x)
    _check(_load().rn_oracle_add_rmsnorm_fmt(_ptr(x, ctypes.c_uint16), _ptr(res, ctypes.c_uint16),
                                             _ptr(w, ctypes.c_uint16), ctypes.c_float(eps), M, N,
                                             _ptr(h, ctypes.c_uint16), _ptr(y, ctypes.c_uint16),
                                             int(f16)), "add_rmsnorm")
    return h, y


def layernorm(x: np.ndarray, w: np.ndarray, b: np.ndarray | None, eps: float,
              f16: bool = False) -> np.ndarray:
    """y = round((x - mean) / sqrt(var + eps) * w + b) row by row (biased
    variance; bf16, or fp16 with f16=True)."""
    x = _u16(x)
    w = _u16(w)
    M, N = x.shape
    y = np.zeros_like(x)
    bp = None if b is None else _ptr(_u16(b), ctypes.c_uint16)
    _check(_load().rn_oracle_layernorm_fmt(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                                           bp, ctypes.c_float(eps), M, N,
                                           _ptr(y, ctypes.c_uint16), int(f16)), "layernorm")
    return y
