"""Performance gate: the stated bandwidth targets, checked on the GPU.

"[pretuned] Optimize fused_qk_norm_rope on B200" ("Tests") pairs its
correctness gate with a performance gate; this is ours.  The targets are
fractions of the measured device copy bandwidth (MEASURED_PEAKS.json
`hbm_gbs`, else the 6800 GB/s fallback figure):

* RMSNorm at M >= 8192 and N >= 8192: at least 0.88, through rmsnorm_fwd_ws
  (the call the bench times: a caller-owned workspace, dynamic unit order);
* fused Q/K RMSNorm + RoPE (Hq 32, Hkv 8, D 128) at T in {4096, 16384},
  rotary 128 and 64, positions uniform in [0, 131072): at least 0.80.

Each launch is timed in steady state: 20 back-to-back launches replayed from
a CUDA graph, alternating two sets of activations (so nothing stays in L2
from one launch to the next), the median replay over about 0.3 s.  The ideal bytes are
counted once (RMSNorm 4MN + 2N; QK 21 000 B a token at rotary 128, 20 744 at
64, plus the weights).  SM clocks are sampled with nvidia-smi meanwhile: a
run with a thermal or hardware slowdown, or clocks well below their maximum,
measures the box rather than the kernels, so it is skipped with the reason.
Set RN_PERF_REPORT to a path to write every figure with its clocks as JSON.
"""
from __future__ import annotations

import json
import os
import statistics

import pytest
import torch

from row_normalization_gb300 import binding, inputs
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RMS_TARGET = 0.88
QK_TARGET = 0.80
FALLBACK_GBS = 6800.0
REPORT: list = []


def peak_gbs() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"])
    except (OSError, ValueError, KeyError):
        return FALLBACK_GBS


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    path = os.environ.get("RN_PERF_REPORT")
    if path and REPORT:
        with open(path, "w") as fh:
            json.dump(REPORT, fh, indent=1)


def steady_ms(launch, reps: int = 20, seconds: float = 0.3) -> float:
    """Milliseconds per launch of launch(i), i = 0..reps-1, replayed from a
    CUDA graph: the median replay over about `seconds` of replays, after one
    warm replay (long enough for the clock sampler to see the load)."""
    import time
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(4):
            launch(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            launch(i)
    g.replay()
    torch.cuda.synchronize()
    times = []
    t_end = time.perf_counter() + seconds
    while len(times) < 3 or time.perf_counter() < t_end:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    del g
    return statistics.median(times)


def measure(label: str, nbytes: int, launch, target: float) -> None:
    from bench import ClockSampler  # nvidia-smi sampler of the bench
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    ms = steady_ms(launch)
    clocks = sampler.stop()
    peak = peak_gbs()
    frac = nbytes / (ms * 1e-3) / 1e9 / peak
    entry = {"case": label, "us": round(ms * 1e3, 2), "frac_of_measured": round(frac, 4),
             "target": target, "peak_gbs": peak, "clocks": clocks}
    REPORT.append(entry)
    if clocks:
        bad = [r for r in clocks["reasons"] if r != "sw_power_cap"]
        if bad or clocks["sm_mhz"] < 0.8 * clocks["sm_max_mhz"]:
            pytest.skip(f"{label}: clocks not at full speed during the timing: {clocks}")
    assert frac >= target, f"{label}: {frac:.3f} of the measured copy < {target}: {entry}"


@pytest.mark.parametrize("M,N", [(8192, 8192), (8192, 16384), (16384, 8192), (16384, 16384),
                                 (32768, 8192), (32768, 16384), (8192, 32768)])
def test_rmsnorm_bandwidth_target(M, N):
    xs = [inputs.rmsnorm_inputs(M, N, outlier_frac=0.01, device="cuda", seed=s)[0]
          for s in (1, 2)]
    w = inputs.norm_weight(N, device="cuda")
    ys = [torch.empty_like(xs[0]) for _ in range(2)]
    ws = binding.new_workspace()
    measure(f"rmsnorm {M}x{N}", 4 * M * N + 2 * N,
            lambda i: binding.rmsnorm_fwd(xs[i & 1], w, 1e-6, ys[i & 1], workspace=ws),
            RMS_TARGET)


@pytest.mark.parametrize("r", [128, 64])
@pytest.mark.parametrize("T", [4096, 16384])
def test_qk_norm_rope_bandwidth_target(T, r):
    table = binding.rope_cos_sin_table(1e6, 131072, r)
    bufs = [inputs.qkv_inputs(T, 32, 8, 128, positions="uniform", max_pos=131072, device="cuda",
                              seed=s) for s in (1, 2)]

    def launch(i):
        q, wq, wk, pos = bufs[i & 1]
        binding.qk_norm_rope_fwd(q, wq, wk, table, pos, 32, 8, 128, r, 1e-6)

    nbytes = T * (2 * 40 * 128 * 2 + r * 4 + 8) + 2 * 128 * 2
    measure(f"qk_norm_rope T={T} r={r}", nbytes, launch, QK_TARGET)
