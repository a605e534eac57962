"""Shared fixtures for the GPU parity tests."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.build import build
from row_normalization_gb300.inputs import bf16_bits


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    binding.load()


@functools.lru_cache(maxsize=8)
def oracle_table(theta: float, max_pos: int, rotary_dim: int) -> np.ndarray:
    return oracle.rope_cos_sin(theta, max_pos, rotary_dim)


def oracle_table_bf16(theta: float, max_pos: int, rotary_dim: int):
    """The oracle's bf16 table twice: as a CUDA bf16 tensor for the library,
    and widened (exactly) to fp32 for the oracle's fused Q/K step."""
    bits = oracle.rope_cos_sin_bf16(theta, max_pos, rotary_dim)
    dev = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    wide = (bits.astype(np.uint32) << 16).view(np.float32)
    return dev, wide


def padded_empty(shape, dtype, pad: int, fill_bits: int):
    """A CUDA tensor of `shape` carved from a larger buffer whose `pad`
    elements on each side are set to a canary bit pattern."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * pad, dtype=torch.int16, device="cuda")
    buf.fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
    view = buf[pad:pad + n].view(dtype).view(*shape)
    return buf, view


def canary_intact(buf: torch.Tensor, pad: int, fill_bits: int) -> bool:
    b = bf16_bits(buf.view(torch.bfloat16))
    return bool(np.all(b[:pad] == fill_bits) and np.all(b[-pad:] == fill_bits))


def bulk_eligible(N: int, mode: str = "rms") -> bool:
    """Whether the persistent bulk-copy schedule serves row width N for
    mode "rms" (RMSNorm, L2Norm), "add" (fused residual add) or "ln"
    (LayerNorm): power-of-two widths 1024..32768 (the fused forms up to
    16384), and any other N % 8 == 0 from 512 up whose generic layout fits."""
    if N % 8 or N < 512 or N > 32768:
        return False
    if N >= 1024 and (N & (N - 1)) == 0:
        return N <= 16384 if mode in ("add", "ln") else True
    cpr = N // 8
    cap = 256 if mode in ("add", "ln") else 512
    vpr = 1
    while vpr < 8 and -(-cpr // vpr) > cap:
        vpr *= 2
    per = -(-cpr // vpr)
    if per > cap:
        return False
    rows = 8 // vpr
    stage = (2 if mode == "add" else 1) * rows * N * 2
    return 2 * stage <= 200 * 1024
