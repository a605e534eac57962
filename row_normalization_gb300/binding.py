"""Thin Python binding over the C ABI of ``librownorm.so`` (include/row_norm.h).

Argument marshalling only: every function checks the tensors' dtype, device
and layout, passes raw pointers, sizes and the current CUDA stream to the
C entry point of the same name, and raises on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.  If the
library is not built, the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

_lock = threading.Lock()
_lib = None

RN_OK = 0
RN_ERR_NULL = -1
RN_ERR_ALIGN = -2
RN_ERR_SHAPE = -3
RN_ERR_LAUNCH = -4
RN_ERR_DEVICE = -5
RN_ERR_ARG = -6

RN_STATUS_WAIT_TIMEOUT = 1
RN_STATUS_BAD_POSITION = 2

RN_SCHED_AUTO = 0
RN_SCHED_WARP_ROW = 1
RN_SCHED_CTA_ROW = 2
RN_SCHED_PERSIST_BULK = 3

RN_QK_AUTO = 0
RN_QK_HEAD_PER_WARP = 1
RN_QK_TWO_HEADS = 2
RN_QK_FOUR_HEADS = 4
RN_QK_PERSISTENT = 8
RN_QK_BULK = 16
RN_QK_PAIRS = 32

RN_ROPE_NEOX = 0
RN_ROPE_GPTJ = 1

RN_DTYPE_BF16 = 0
RN_DTYPE_F16 = 1

RN_OP_RMSNORM = 0
RN_OP_L2NORM = 1
RN_OP_ADD_RMSNORM = 2
RN_OP_LAYERNORM = 3

RN_WORKSPACE_BYTES = 256
RN_NOALLOC_SCRATCH_BYTES = 256  # the fixed scratch array of rmsnorm_fwd_noalloc

_ROW_DTYPES = {torch.bfloat16: RN_DTYPE_BF16, torch.float16: RN_DTYPE_F16}


class RowNormError(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__(f"{name}: {error_string(code)} (status {code})")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once).  Raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(row_normalization_gb300.build.build())")
        L = ctypes.CDLL(path)
        vp, i64, i32, f32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_double)
        u64 = ctypes.c_uint64
        L.rn_error_string.argtypes = [i32]
        L.rn_error_string.restype = ctypes.c_char_p
        L.rn_version.argtypes = []
        L.rn_version.restype = i32
        L.rmsnorm_fwd.argtypes = [vp, vp, f32, i64, i64, vp, vp]
        L.rmsnorm_fwd.restype = i32
        L.rmsnorm_fwd_sched.argtypes = [vp, vp, f32, i64, i64, vp, i32, u64, i32, vp]
        L.rmsnorm_fwd_sched.restype = i32
        L.qk_norm_rope_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, vp]
        L.qk_norm_rope_fwd.restype = i32
        L.qk_norm_rope_fwd_sched.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32,
                                             i32, u64, i32, vp]
        L.qk_norm_rope_fwd_sched.restype = i32
        L.qk_norm_rope_fwd_checked.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32,
                                               i64, vp, vp]
        L.qk_norm_rope_fwd_checked.restype = i32
        L.qk_norm_rope_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, i32,
                                          i64, vp, i32, u64, i32, vp]
        L.qk_norm_rope_fwd_ex.restype = i32
        L.rope_cos_sin_table.argtypes = [f64, i64, i32, vp, vp]
        L.rope_cos_sin_table.restype = i32
        L.qk_norm_rope_fwd_ex_bf16_table.argtypes = L.qk_norm_rope_fwd_ex.argtypes
        L.qk_norm_rope_fwd_ex_bf16_table.restype = i32
        L.rope_cos_sin_table_bf16.argtypes = [f64, i64, i32, vp, vp]
        L.rope_cos_sin_table_bf16.restype = i32
        L.rope_cos_sin_table_host.argtypes = [f64, i64, i32, vp]
        L.rope_cos_sin_table_host.restype = i32
        L.rmsnorm_fwd_ws.argtypes = [vp, vp, f32, i64, i64, vp, vp, vp]
        L.rmsnorm_fwd_ws.restype = i32
        L.row_norm_fwd_ws.argtypes = [i32, i32, vp, vp, vp, vp, f32, i64, i64, vp, vp, vp, i32,
                                      u64, i32, vp]
        L.row_norm_fwd_ws.restype = i32
        L.rmsnorm_fwd_noalloc.argtypes = [vp, vp, f32, i64, i64, vp, vp]
        L.rmsnorm_fwd_noalloc.restype = i32
        L.add_rmsnorm_fwd.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp, vp]
        L.add_rmsnorm_fwd.restype = i32
        L.add_rmsnorm_fwd_sched.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp, i32, u64, i32, vp]
        L.add_rmsnorm_fwd_sched.restype = i32
        L.l2norm_fwd.argtypes = [vp, f32, i64, i64, vp, vp]
        L.l2norm_fwd.restype = i32
        L.l2norm_fwd_sched.argtypes = [vp, f32, i64, i64, vp, i32, u64, i32, vp]
        L.l2norm_fwd_sched.restype = i32
        L.layernorm_fwd.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp]
        L.layernorm_fwd.restype = i32
        L.layernorm_fwd_sched.argtypes = [vp, vp, vp, f32, i64, i64, vp, i32, u64, i32, vp]
        L.layernorm_fwd_sched.restype = i32
        L.layernorm_select_schedule.argtypes = [i64, i64]
        L.layernorm_select_schedule.restype = i32
        L.add_rmsnorm_select_schedule.argtypes = [i64, i64]
        L.add_rmsnorm_select_schedule.restype = i32
        L.rmsnorm_select_schedule.argtypes = [i64, i64]
        L.rmsnorm_select_schedule.restype = i32
        L.qk_norm_rope_select_schedule.argtypes = [i64]
        L.qk_norm_rope_select_schedule.restype = i32
        L.qk_norm_rope_select_schedule_ex.argtypes = [i64, i32, i32]
        L.qk_norm_rope_select_schedule_ex.restype = i32
        L.rmsnorm_fwd_f16.argtypes = [vp, vp, f32, i64, i64, vp, vp]
        L.rmsnorm_fwd_f16.restype = i32
        L.l2norm_fwd_f16.argtypes = [vp, f32, i64, i64, vp, vp]
        L.l2norm_fwd_f16.restype = i32
        L.add_rmsnorm_fwd_f16.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp, vp]
        L.add_rmsnorm_fwd_f16.restype = i32
        L.layernorm_fwd_f16.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp]
        L.layernorm_fwd_f16.restype = i32
        L.row_norm_fwd_ex.argtypes = [i32, i32, vp, vp, vp, vp, f32, i64, i64, vp, vp, i32, u64,
                                      i32, vp]
        L.row_norm_fwd_ex.restype = i32
        L.row_norm_select_schedule.argtypes = [i32, i64, i64]
        L.row_norm_select_schedule.restype = i32
        L.row_norm_select_schedule_ws.argtypes = [i32, i64, i64]
        L.row_norm_select_schedule_ws.restype = i32
        L.rn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        L.rn_device_status.restype = i32
        _lib = L
        return L


def error_string(code: int) -> str:
    return load().rn_error_string(int(code)).decode()


def version() -> int:
    return int(load().rn_version())


def _check(rc: int, name: str) -> None:
    if rc != RN_OK:
        raise RowNormError(name, rc)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _row_dtype(x: torch.Tensor) -> torch.dtype:
    """The element format of a row-norm call: x's dtype, bf16 or fp16."""
    if not isinstance(x, torch.Tensor):
        raise TypeError("x must be a torch.Tensor")
    if x.dtype not in _ROW_DTYPES:
        raise TypeError(f"x must be torch.bfloat16 or torch.float16, got {x.dtype}")
    return x.dtype


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _row_ex(name, op, dt, x, r, w, b, eps, M, N, h, y, schedule, wait_timeout_ns, debug_flags,
            stream):
    rc = load().row_norm_fwd_ex(op, _ROW_DTYPES[dt], _ptr(x), _ptr(r), _ptr(w), _ptr(b), eps, M,
                                N, _ptr(h), _ptr(y), schedule, wait_timeout_ns, debug_flags,
                                _stream(stream))
    _check(rc, name)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def new_workspace(device=None) -> torch.Tensor:
    """A zeroed workspace for the *_ws entry points (RN_WORKSPACE_BYTES of
    device memory).  Calls that run one after another (one stream) can share
    one; calls that may run at the same time need one each."""
    return torch.zeros(RN_WORKSPACE_BYTES, dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _ws(workspace: torch.Tensor | None):
    """Device pointer of a caller's workspace (checked), or None."""
    if workspace is None:
        return None
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if not workspace.is_contiguous() or \
            workspace.numel() * workspace.element_size() < RN_WORKSPACE_BYTES:
        raise ValueError(f"workspace must be a contiguous tensor of >= {RN_WORKSPACE_BYTES} bytes")
    return workspace.data_ptr()


def _row_ws(name, op, dt, x, r, w, b, eps, M, N, h, y, workspace, schedule, wait_timeout_ns,
            debug_flags, stream):
    rc = load().row_norm_fwd_ws(op, _ROW_DTYPES[dt], _ptr(x), _ptr(r), _ptr(w), _ptr(b), eps, M,
                                N, _ptr(h), _ptr(y), _ws(workspace), schedule, wait_timeout_ns,
                                debug_flags, _stream(stream))
    _check(rc, name)


# ---------------------------------------------------------------------------

def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float, y: torch.Tensor | None = None,
                *, schedule: int = RN_SCHED_AUTO, wait_timeout_ns: int = 0,
                debug_flags: int = 0, stream=None,
                workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y = x * rsqrt(mean(x^2, -1) + eps) * w for x [M, N] in bf16 or fp16
    (w and y in x's dtype); returns y.  With a `workspace` (new_workspace())
    the persistent schedule takes its units in the dynamic order."""
    dt = _row_dtype(x)
    _need(x, "x", dt)
    _need(w, "w", dt)
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("x must be [M, N] and w [N]")
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", dt)
        if y.shape != x.shape:
            raise ValueError("y must have x's shape")
    M, N = x.shape
    L = load()
    plain = schedule == RN_SCHED_AUTO and wait_timeout_ns == 0 and debug_flags == 0
    if workspace is not None:
        if plain and dt == torch.bfloat16:
            _check(L.rmsnorm_fwd_ws(x.data_ptr(), w.data_ptr(), eps, M, N, y.data_ptr(),
                                    _ws(workspace), _stream(stream)), "rmsnorm_fwd_ws")
        else:
            _row_ws("row_norm_fwd_ws", RN_OP_RMSNORM, dt, x, None, w, None, eps, M, N, None, y,
                    workspace, schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if dt == torch.float16:
        if plain:
            _check(L.rmsnorm_fwd_f16(x.data_ptr(), w.data_ptr(), eps, M, N, y.data_ptr(),
                                     _stream(stream)), "rmsnorm_fwd_f16")
        else:
            _row_ex("row_norm_fwd_ex", RN_OP_RMSNORM, dt, x, None, w, None, eps, M, N, None, y,
                    schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if plain:
        rc = L.rmsnorm_fwd(x.data_ptr(), w.data_ptr(), eps, M, N, y.data_ptr(), _stream(stream))
    else:
        rc = L.rmsnorm_fwd_sched(x.data_ptr(), w.data_ptr(), eps, M, N, y.data_ptr(),
                                 schedule, wait_timeout_ns, debug_flags, _stream(stream))
    _check(rc, "rmsnorm_fwd")
    return y


def rmsnorm_fwd_noalloc(x: torch.Tensor, w: torch.Tensor, eps: float,
                        y: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """rmsnorm_fwd (bf16) for callers that cannot allocate device memory: the
    library's own scratch array replaces the workspace.  Calls that may run at
    the same time on one GPU race on that array; see include/row_norm.h."""
    _need(x, "x", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("x must be [M, N] and w [N]")
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", torch.bfloat16)
        if y.shape != x.shape:
            raise ValueError("y must have x's shape")
    M, N = x.shape
    _check(load().rmsnorm_fwd_noalloc(x.data_ptr(), w.data_ptr(), eps, M, N, y.data_ptr(),
                                      _stream(stream)), "rmsnorm_fwd_noalloc")
    return y


def l2norm_fwd(x: torch.Tensor, eps: float, y: torch.Tensor | None = None, *,
               schedule: int = RN_SCHED_AUTO, wait_timeout_ns: int = 0, debug_flags: int = 0,
               stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y = x / max(||x||_2, eps) per row of x [M, N] (bf16 or fp16)."""
    dt = _row_dtype(x)
    _need(x, "x", dt)
    if x.dim() != 2:
        raise ValueError("x must be [M, N]")
    y = torch.empty_like(x) if y is None else y
    _need(y, "y", dt)
    if y.shape != x.shape:
        raise ValueError("y must have x's shape")
    M, N = x.shape
    L = load()
    plain = schedule == RN_SCHED_AUTO and wait_timeout_ns == 0 and debug_flags == 0
    if workspace is not None:
        _row_ws("row_norm_fwd_ws", RN_OP_L2NORM, dt, x, None, None, None, eps, M, N, None, y,
                workspace, schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if dt == torch.float16:
        if plain:
            _check(L.l2norm_fwd_f16(x.data_ptr(), eps, M, N, y.data_ptr(), _stream(stream)),
                   "l2norm_fwd_f16")
        else:
            _row_ex("row_norm_fwd_ex", RN_OP_L2NORM, dt, x, None, None, None, eps, M, N, None, y,
                    schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if plain:
        rc = L.l2norm_fwd(x.data_ptr(), eps, M, N, y.data_ptr(), _stream(stream))
    else:
        rc = L.l2norm_fwd_sched(x.data_ptr(), eps, M, N, y.data_ptr(), schedule,
                                wait_timeout_ns, debug_flags, _stream(stream))
    _check(rc, "l2norm_fwd")
    return y


def layernorm_fwd(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor | None, eps: float,
                  y: torch.Tensor | None = None, *, schedule: int = RN_SCHED_AUTO,
                  wait_timeout_ns: int = 0, debug_flags: int = 0, stream=None,
                  workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y = (x - mean) / sqrt(var + eps) * w + b per row (biased variance); b may
    be None.  bf16 or fp16, every tensor in x's dtype."""
    dt = _row_dtype(x)
    _need(x, "x", dt)
    _need(w, "w", dt)
    if b is not None:
        _need(b, "b", dt)
        if b.shape != w.shape:
            raise ValueError("b must have w's shape")
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("x must be [M, N] and w [N]")
    y = torch.empty_like(x) if y is None else y
    _need(y, "y", dt)
    if y.shape != x.shape:
        raise ValueError("y must have x's shape")
    M, N = x.shape
    bp = None if b is None else b.data_ptr()
    L = load()
    plain = schedule == RN_SCHED_AUTO and wait_timeout_ns == 0 and debug_flags == 0
    if workspace is not None:
        _row_ws("row_norm_fwd_ws", RN_OP_LAYERNORM, dt, x, None, w, b, eps, M, N, None, y,
                workspace, schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if dt == torch.float16:
        if plain:
            _check(L.layernorm_fwd_f16(x.data_ptr(), w.data_ptr(), bp, eps, M, N, y.data_ptr(),
                                       _stream(stream)), "layernorm_fwd_f16")
        else:
            _row_ex("row_norm_fwd_ex", RN_OP_LAYERNORM, dt, x, None, w, b, eps, M, N, None, y,
                    schedule, wait_timeout_ns, debug_flags, stream)
        return y
    if plain:
        rc = L.layernorm_fwd(x.data_ptr(), w.data_ptr(), bp, eps, M, N, y.data_ptr(),
                             _stream(stream))
    else:
        rc = L.layernorm_fwd_sched(x.data_ptr(), w.data_ptr(), bp, eps, M, N, y.data_ptr(),
                                   schedule, wait_timeout_ns, debug_flags, _stream(stream))
    _check(rc, "layernorm_fwd")
    return y


def row_norm_select_schedule(op: int, M: int, N: int, *, workspace: bool = False) -> int:
    """The RN_SCHED_* schedule a row norm (RN_OP_*) picks for (M, N); the same
    for both element formats.  workspace=True: the choice of the workspace
    forms (the dynamic unit order is open to the ring)."""
    name = "row_norm_select_schedule_ws" if workspace else "row_norm_select_schedule"
    rc = int(getattr(load(), name)(int(op), int(M), int(N)))
    if rc < 0:
        raise RowNormError(name, rc)
    return rc


def layernorm_select_schedule(M: int, N: int) -> int:
    """The RN_SCHED_* schedule layernorm_fwd picks for (M, N) on the current device."""
    rc = int(load().layernorm_select_schedule(int(M), int(N)))
    if rc < 0:
        raise RowNormError("layernorm_select_schedule", rc)
    return rc


def add_rmsnorm_fwd(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor, eps: float,
                    h: torch.Tensor | None = None, y: torch.Tensor | None = None, *,
                    schedule: int = RN_SCHED_AUTO, wait_timeout_ns: int = 0,
                    debug_flags: int = 0, stream=None, workspace: torch.Tensor | None = None):
    """h = x + residual, y = rmsnorm(h); returns (h, y).  bf16 or fp16, every
    tensor in x's dtype.  Pass h=residual for an in-place residual update."""
    dt = _row_dtype(x)
    _need(x, "x", dt)
    _need(residual, "residual", dt)
    _need(w, "w", dt)
    if x.dim() != 2 or residual.shape != x.shape or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("x and residual must be [M, N] and w [N]")
    h = torch.empty_like(x) if h is None else h
    y = torch.empty_like(x) if y is None else y
    _need(h, "h", dt)
    _need(y, "y", dt)
    if h.shape != x.shape or y.shape != x.shape:
        raise ValueError("h and y must have x's shape")
    M, N = x.shape
    L = load()
    plain = schedule == RN_SCHED_AUTO and wait_timeout_ns == 0 and debug_flags == 0
    if workspace is not None:
        _row_ws("row_norm_fwd_ws", RN_OP_ADD_RMSNORM, dt, x, residual, w, None, eps, M, N, h, y,
                workspace, schedule, wait_timeout_ns, debug_flags, stream)
        return h, y
    if dt == torch.float16:
        if plain:
            _check(L.add_rmsnorm_fwd_f16(x.data_ptr(), residual.data_ptr(), w.data_ptr(), eps, M,
                                         N, h.data_ptr(), y.data_ptr(), _stream(stream)),
                   "add_rmsnorm_fwd_f16")
        else:
            _row_ex("row_norm_fwd_ex", RN_OP_ADD_RMSNORM, dt, x, residual, w, None, eps, M, N, h,
                    y, schedule, wait_timeout_ns, debug_flags, stream)
        return h, y
    if plain:
        rc = L.add_rmsnorm_fwd(x.data_ptr(), residual.data_ptr(), w.data_ptr(), eps, M, N,
                               h.data_ptr(), y.data_ptr(), _stream(stream))
    else:
        rc = L.add_rmsnorm_fwd_sched(x.data_ptr(), residual.data_ptr(), w.data_ptr(), eps, M, N,
                                     h.data_ptr(), y.data_ptr(), schedule, wait_timeout_ns,
                                     debug_flags, _stream(stream))
    _check(rc, "add_rmsnorm_fwd")
    return h, y


def _qk_common(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim):
    _need(qkv, "qkv", torch.bfloat16)
    _need(wq, "wq", torch.bfloat16)
    _need(wk, "wk", torch.bfloat16)
    # the table may hold fp32 or bf16 entries (the bf16 form has its own entry point)
    _need(cos_sin, "cos_sin", torch.bfloat16 if cos_sin.dtype == torch.bfloat16 else torch.float32)
    _need(positions, "positions", torch.int64)
    T = qkv.shape[0]
    if qkv.numel() != T * (Hq + 2 * Hkv) * D:
        raise ValueError("qkv must be [T, (Hq + 2*Hkv) * D]")
    if wq.numel() != D or wk.numel() != D:
        raise ValueError("wq and wk must have D elements")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != rotary_dim:
        raise ValueError("cos_sin must be [max_pos, rotary_dim]")
    if positions.numel() != T:
        raise ValueError("positions must have T elements")
    return T


def qk_norm_rope_fwd(qkv: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor,
                     cos_sin: torch.Tensor, positions: torch.Tensor, Hq: int, Hkv: int, D: int,
                     rotary_dim: int, eps: float, *, schedule: int = RN_QK_AUTO,
                     wait_timeout_ns: int = 0, debug_flags: int = 0,
                     stream=None) -> torch.Tensor:
    """In place: per-head RMSNorm of Q and K heads, then neox RoPE.  Returns qkv."""
    T = _qk_common(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim)
    L = load()
    if cos_sin.dtype == torch.bfloat16:
        return _qk_bf16_table(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                              RN_ROPE_NEOX, 0, None, schedule, wait_timeout_ns, debug_flags,
                              stream, "qk_norm_rope_fwd")
    if schedule == RN_QK_AUTO and wait_timeout_ns == 0 and debug_flags == 0:
        rc = L.qk_norm_rope_fwd(qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(), cos_sin.data_ptr(),
                                positions.data_ptr(), T, Hq, Hkv, D, rotary_dim, eps,
                                _stream(stream))
    else:
        rc = L.qk_norm_rope_fwd_sched(qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                      cos_sin.data_ptr(), positions.data_ptr(), T, Hq, Hkv, D,
                                      rotary_dim, eps, schedule, wait_timeout_ns, debug_flags,
                                      _stream(stream))
    _check(rc, "qk_norm_rope_fwd")
    return qkv


def _qk_bf16_table(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps, style,
                   max_pos, err_ptr, schedule, wait_timeout_ns, debug_flags, stream, what):
    rc = load().qk_norm_rope_fwd_ex_bf16_table(
        qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(), cos_sin.data_ptr(), positions.data_ptr(), T,
        Hq, Hkv, D, rotary_dim, eps, style, int(max_pos), err_ptr, schedule, wait_timeout_ns,
        debug_flags, _stream(stream))
    _check(rc, what)
    return qkv


def qk_norm_rope_fwd_ex(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim, eps, *,
                        rope_style: int = RN_ROPE_NEOX, max_pos: int = 0,
                        err_flag: torch.Tensor | None = None, schedule: int = RN_QK_AUTO,
                        wait_timeout_ns: int = 0, debug_flags: int = 0, stream=None):
    """The general QK entry: rope_style (neox / GPT-J), optional position checks
    (max_pos > 0 with an int32 CUDA err_flag), schedule and test flags."""
    T = _qk_common(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim)
    ep = None
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
        ep = err_flag.data_ptr()
    if cos_sin.dtype == torch.bfloat16:
        return _qk_bf16_table(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                              rope_style, max_pos, ep, schedule, wait_timeout_ns, debug_flags,
                              stream, "qk_norm_rope_fwd_ex")
    rc = load().qk_norm_rope_fwd_ex(qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                    cos_sin.data_ptr(), positions.data_ptr(), T, Hq, Hkv, D,
                                    rotary_dim, eps, rope_style, int(max_pos), ep, schedule,
                                    wait_timeout_ns, debug_flags, _stream(stream))
    _check(rc, "qk_norm_rope_fwd_ex")
    return qkv


def qk_norm_rope_fwd_checked(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim, eps,
                             err_flag: torch.Tensor, *, max_pos: int | None = None,
                             stream=None) -> torch.Tensor:
    """As qk_norm_rope_fwd; tokens with a position outside [0, max_pos) are left
    untouched and RN_STATUS_BAD_POSITION is OR-ed into err_flag (int32 CUDA [1])."""
    T = _qk_common(qkv, wq, wk, cos_sin, positions, Hq, Hkv, D, rotary_dim)
    _need(err_flag, "err_flag", torch.int32)
    if max_pos is None:
        max_pos = cos_sin.shape[0]
    if cos_sin.dtype == torch.bfloat16:
        if int(max_pos) < 1:
            raise RowNormError("qk_norm_rope_fwd_checked", RN_ERR_SHAPE)
        return _qk_bf16_table(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                              RN_ROPE_NEOX, max_pos, err_flag.data_ptr(), RN_QK_AUTO, 0, 0,
                              stream, "qk_norm_rope_fwd_checked")
    rc = load().qk_norm_rope_fwd_checked(qkv.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                                         cos_sin.data_ptr(), positions.data_ptr(), T, Hq, Hkv, D,
                                         rotary_dim, eps, int(max_pos), err_flag.data_ptr(),
                                         _stream(stream))
    _check(rc, "qk_norm_rope_fwd_checked")
    return qkv


def rope_cos_sin_table(theta: float, max_pos: int, rotary_dim: int,
                       out: torch.Tensor | None = None, *, device=None,
                       dtype: torch.dtype | None = None, stream=None) -> torch.Tensor:
    """[max_pos, rotary_dim] table: cos half then sin half of p * theta^(-2i/r),
    fp32 (default) or bf16 (dtype=torch.bfloat16, or a bf16 `out`), each entry
    rounded once from fp64.  Built on the GPU into a CUDA tensor; with
    device="cpu" (or a CPU `out`) an fp32 table is built by the library's host
    form (rope_cos_sin_table_host) into host memory."""
    if dtype is None:
        dtype = out.dtype if out is not None else torch.float32
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("rope_cos_sin_table builds fp32 or bf16 tables")
    on_host = (out is not None and out.device.type == "cpu") or \
        (out is None and device is not None and torch.device(device).type == "cpu")
    if on_host:
        if dtype != torch.float32:
            raise TypeError("the host table builder writes fp32 entries")
        if out is None:
            out = torch.empty(max_pos, rotary_dim, dtype=torch.float32)
        if out.shape != (max_pos, rotary_dim) or not out.is_contiguous():
            raise ValueError("out must be a contiguous [max_pos, rotary_dim] tensor")
        rc = load().rope_cos_sin_table_host(float(theta), int(max_pos), int(rotary_dim),
                                            out.data_ptr())
        _check(rc, "rope_cos_sin_table_host")
        return out
    if out is None:
        out = torch.empty(max_pos, rotary_dim, dtype=dtype,
                          device=device if device is not None else "cuda")
    _need(out, "out", dtype)
    if out.shape != (max_pos, rotary_dim):
        raise ValueError("out must be [max_pos, rotary_dim]")
    L = load()
    fn = L.rope_cos_sin_table_bf16 if dtype == torch.bfloat16 else L.rope_cos_sin_table
    rc = fn(float(theta), int(max_pos), int(rotary_dim), out.data_ptr(), _stream(stream))
    _check(rc, "rope_cos_sin_table")
    return out


def rmsnorm_select_schedule(M: int, N: int, *, workspace: bool = False) -> int:
    """The RN_SCHED_* schedule rmsnorm_fwd picks for (M, N) on the current
    device; workspace=True: the schedule of rmsnorm_fwd with a workspace."""
    if workspace:
        return row_norm_select_schedule(RN_OP_RMSNORM, M, N, workspace=True)
    rc = int(load().rmsnorm_select_schedule(int(M), int(N)))
    if rc < 0:
        raise RowNormError("rmsnorm_select_schedule", rc)
    return rc


def add_rmsnorm_select_schedule(M: int, N: int) -> int:
    """The RN_SCHED_* schedule add_rmsnorm_fwd picks for (M, N) on the current device."""
    rc = int(load().add_rmsnorm_select_schedule(int(M), int(N)))
    if rc < 0:
        raise RowNormError("add_rmsnorm_select_schedule", rc)
    return rc


def qk_norm_rope_select_schedule(T: int, head_dim: int = 128, rotary_dim: int = 128) -> int:
    """The RN_QK_* schedule qk_norm_rope_fwd picks for T tokens of this layout."""
    rc = int(load().qk_norm_rope_select_schedule_ex(int(T), int(head_dim), int(rotary_dim)))
    if rc < 0:
        raise RowNormError("qk_norm_rope_select_schedule_ex", rc)
    return rc


def device_status(clear: bool = True) -> int:
    """OR of RN_STATUS_* bits raised on the current device (synchronises)."""
    v = ctypes.c_uint(0)
    _check(load().rn_device_status(ctypes.byref(v), 1 if clear else 0), "rn_device_status")
    return int(v.value)
