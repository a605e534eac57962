"""Seeded synthetic inputs for row normalization (bf16, or fp16 for the row norms).

This module only draws random numbers; it holds none of the normalisation
or rotary arithmetic.  The same tensors feed the CUDA library and the CPU
oracle.  Every distribution follows the workloads the pages measure:

* RMSNorm rows: x ~ N(0, 1), optionally with a fraction of rows scaled by
  100 (outlier rows) in fp32 before the bf16 rounding; weight
  w = 1 + 0.1 * N(0, 1).  Sizes come from the caller (M rows of N).
* Packed QKV: every element ~ N(0, 1); q and k norm weights
  1 + 0.1 * N(0, 1); positions either 0..T-1 or uniform in [0, max_pos).

Seeds: x / qkv = seed, w / wq = seed + 1, outlier rows = seed + 2,
wk = seed + 3, positions = seed + 4.  fp32 draws are rounded to the element
format (bf16 by default, or ``dtype=torch.float16``) with round-to-nearest-even
(``Tensor.to``); the fp16 draws are the same fp32 numbers rounded to fp16.

``device="cuda"`` draws on the GPU (torch's Philox generator), which the
large workloads need; ``device="cpu"`` draws on the host.  The two devices
give different numbers for the same seed; a caller compares the CUDA library
and the oracle on the same tensor, never across devices.
"""
from __future__ import annotations

import torch


def _gen(device, seed: int) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def rmsnorm_inputs(M: int, N: int, *, outlier_frac: float = 0.0, device="cpu",
                   seed: int = 0, dtype: torch.dtype = torch.bfloat16):
    """Return (x [M, N], w [N]) in ``dtype`` on ``device``."""
    x = torch.randn(M, N, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    k = int(round(outlier_frac * M))
    if k > 0:
        rows = torch.randperm(M, generator=_gen("cpu", seed + 2))[:k]
        x[rows.to(x.device)] *= 100.0
    x = x.to(dtype)
    w = norm_weight(N, device=device, seed=seed + 1, dtype=dtype)
    return x, w


def norm_weight(n: int, *, device="cpu", seed: int = 1,
                dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """w = 1 + 0.1 * N(0, 1), rounded to ``dtype``."""
    g = torch.randn(n, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return (1.0 + 0.1 * g).to(dtype)


def norm_bias(n: int, *, device="cpu", seed: int = 5,
              dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """b = 0.1 * N(0, 1), rounded to ``dtype`` (LayerNorm's affine shift)."""
    g = torch.randn(n, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return (0.1 * g).to(dtype)


def qkv_inputs(T: int, Hq: int, Hkv: int, D: int, *, positions: str = "arange",
               max_pos: int | None = None, device="cpu", seed: int = 0):
    """Return (qkv [T, (Hq+2*Hkv)*D] bf16, wq [D], wk [D], positions [T] int64).

    ``positions="arange"`` gives 0..T-1; ``"uniform"`` draws uniformly from
    [0, max_pos).
    """
    width = (Hq + 2 * Hkv) * D
    qkv = torch.randn(T, width, generator=_gen(device, seed), device=device,
                      dtype=torch.float32).to(torch.bfloat16)
    wq = norm_weight(D, device=device, seed=seed + 1)
    wk = norm_weight(D, device=device, seed=seed + 3)
    if positions == "arange":
        pos = torch.arange(T, device=device, dtype=torch.int64)
    elif positions == "uniform":
        if not max_pos:
            raise ValueError("uniform positions need max_pos")
        pos = torch.randint(0, int(max_pos), (T,), generator=_gen(device, seed + 4),
                            device=device, dtype=torch.int64)
    else:
        raise ValueError(f"unknown positions mode {positions!r}")
    return qkv, wq, wk, pos


def bf16_bits(t: torch.Tensor):
    """16-bit (bf16 or fp16) tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def bf16_from_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
