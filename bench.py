#!/usr/bin/env python3
"""Throughput of the bf16 row-normalization hot path on one GB300 (or N replicas).

One step = one pass of the whole path over resident synthetic inputs:
  * RMSNorm over the sweep M in {4096, 8192, 16384, 32768} x N in {4096, 8192,
    16384} (x ~ N(0,1) with 1% of rows scaled x100, w = 1 + 0.1 N(0,1),
    eps 1e-6): 12 launches;
  * fused Q/K RMSNorm + neox RoPE on packed QKV [16384, 48*128] (32 query and
    8 key/value heads of 128, theta 1e6, positions uniform in [0, 131072)),
    once with rotary_dim 128 and once with 64: 2 launches.
The metric is achieved HBM bandwidth over the ideal bytes (each input read
once, each output written once), in GB/s, whole job.  Device-side timing
uses CUDA events on the launching stream; `e2e` repeats the step through the
same C entry points with the inputs copied in from pinned host memory and
the outputs copied back inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --impl reference the CPU oracle (the plain fp64 implementation the tests
use as the yardstick) is timed on the host cores on a bounded sample of the
same workload.  Under torchrun with N > 1 every rank runs the same per-GPU
workload (weak scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak for bf16 RMSNorm / QK-norm+RoPE"
SPEC_GBS = 7928.0
L2_BYTES = 126 * 2**20

RMS_SHAPES = [(M, N) for M in (4096, 8192, 16384, 32768) for N in (4096, 8192, 16384)]
ADD_SHAPES: list = []   # fused residual add + RMSNorm: only with --only add:MxN
LN_SHAPES: list = []    # LayerNorm (with bias): only with --only ln:MxN
L2_SHAPES: list = []    # L2Norm: only with --only l2:MxN
ROW_DTYPE = "bf16"      # element format of the row norms (--row-dtype f16 for fp16)
QK_TABLE = "f32"        # element type of the rotary cos/sin table (--qk-table bf16)
RMS_EPS = 1e-6
QK_T = 16384
QK_ROT = (128, 64)
HQ, HKV, D = 32, 8, 128
MAX_POS = 131072
THETA = 1e6
QK_EPS = 1e-6
WORKLOAD = ("rmsnorm sweep M{4096,8192,16384,32768}xN{4096,8192,16384} (1% outlier rows) + "
            "qk_norm_rope T=16384 Hq=32 Hkv=8 D=128 rotary {128,64}")


def rms_bytes(M: int, N: int) -> int:
    """Ideal bytes: read x once, read w once, write y once."""
    return 4 * M * N + 2 * N


def qk_bytes(T: int, r: int) -> int:
    """Ideal bytes: read+write every Q/K head (V untouched), one cos/sin row
    (fp32, or bf16 with --qk-table bf16) and one int64 position per token,
    both weights once."""
    return T * (2 * (HQ + HKV) * D * 2 + r * (2 if QK_TABLE == "bf16" else 4) + 8) + 2 * D * 2


def qk_v_bytes(T: int) -> int:
    """The V heads' bytes if they were read and written too (the count that
    treats QKV as moved in and out whole): reported beside the ideal count."""
    return T * HKV * D * 2 * 2


def add_bytes(M: int, N: int) -> int:
    """Ideal bytes of the fused residual add: read x and r, write h and y, w once."""
    return 8 * M * N + 2 * N


def ln_bytes(M: int, N: int) -> int:
    """Ideal bytes of LayerNorm: read x, write y, w and b once."""
    return 4 * M * N + 4 * N


def l2_bytes(M: int, N: int) -> int:
    """Ideal bytes of L2Norm: read x, write y (no weight)."""
    return 4 * M * N


def step_bytes() -> int:
    return (sum(rms_bytes(M, N) for M, N in RMS_SHAPES) + sum(qk_bytes(QK_T, r) for r in QK_ROT)
            + sum(add_bytes(M, N) for M, N in ADD_SHAPES)
            + sum(ln_bytes(M, N) for M, N in LN_SHAPES)
            + sum(l2_bytes(M, N) for M, N in L2_SHAPES))


def restrict_workload(spec: str) -> None:
    """--only: keep a subset of the step, e.g. "rms:8192x16384,qk:16384:128",
    or measure the fused residual add with "add:8192x8192" (likewise "ln:"
    for LayerNorm, "l2:" for L2Norm).  Used for profiling one launch; the
    printed line names the reduced workload."""
    global RMS_SHAPES, QK_ROT, QK_T, WORKLOAD, ADD_SHAPES, LN_SHAPES, L2_SHAPES
    rms, rot, add, ln, l2 = [], [], [], [], []
    for item in spec.split(","):
        kind, _, rest = item.partition(":")
        if kind == "rms":
            M, N = rest.split("x")
            rms.append((int(M), int(N)))
        elif kind == "qk":
            T, r = rest.split(":")
            QK_T = int(T)
            rot.append(int(r))
        elif kind == "add":
            M, N = rest.split("x")
            add.append((int(M), int(N)))
        elif kind == "ln":
            M, N = rest.split("x")
            ln.append((int(M), int(N)))
        elif kind == "l2":
            M, N = rest.split("x")
            l2.append((int(M), int(N)))
        else:
            raise SystemExit(f"bad --only item {item!r}")
    RMS_SHAPES, QK_ROT, ADD_SHAPES, LN_SHAPES, L2_SHAPES = rms, tuple(rot), add, ln, l2
    WORKLOAD = "subset: " + spec


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return {}


def max_over_ranks(torch, dist, ms: float, device) -> float:
    """The slowest rank's time: every rank ends with the max (NCCL on the GPU
    box, gloo in the CPU tests)."""
    if not dist:
        return ms
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_rank: int, ms: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_rank (replicas: weak scaling)
    in the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] is None or r["power"] > 200.0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"),
                              ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in busy),
                "reasons": sorted(reasons), "samples": len(busy)}


COUNTERS_FILE = os.path.join(ROOT, "profiles", "dram_counters.txt")


def code_only(src: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of
    whitespace made one space: what the compiler sees, so that editing a
    comment does not change a kernel's digest.  String and character literals
    (inline PTX) are kept as written."""
    out = []
    i, n = 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest(kernel: str) -> str:
    """sha256[:16] of the code a kernel is compiled from (its file and the
    shared device helpers, comments and spacing aside), which keys the
    recorded ncu counters."""
    csrc = os.path.join(ROOT, "row_normalization_gb300", "csrc")
    files = ["row_kernels.cuh" if kernel.startswith("rms") else "qk_norm_rope.cu",
             "rn_common.cuh"]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_counters(kernel: str, workload: str):
    """The ncu DRAM counters recorded for one launch (profiles/dram_counters.txt):
    dram__bytes_read.sum, dram__bytes_write.sum and
    dram__throughput.avg.pct_of_peak_sustained_elapsed, or None when no
    capture matches or the kernel's sources changed since it was taken."""
    try:
        digest = kernel_source_digest(kernel)
        with open(COUNTERS_FILE) as fh:
            for line in fh:
                if line.startswith("#") or "|" not in line:
                    continue
                k, wl, rd, wr, pct, sha = [p.strip() for p in line.split("|")[:6]]
                if k == kernel and wl == workload and sha == digest:
                    return {"dram_bytes_read": int(float(rd)), "dram_bytes_write": int(float(wr)),
                            "dram_throughput_pct_of_peak": float(pct),
                            "source": "profiles/dram_counters.txt (ncu, one pass, cold caches)"}
    except OSError:
        return None
    return None


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

RMS_KERNELS = {1: "rms_warp_rows_kernel", 2: "rms_cta_rows_kernel", 3: "rms_persistent_bulk_kernel"}
QK_KERNELS = {1: "qk_norm_rope_kernel", 2: "qk_norm_rope_kernel", 4: "qk_norm_rope_kernel",
              8: "qk_norm_rope_kernel", 16: "qk_persistent_bulk_kernel", 32: "qk_pair_kernel"}


def table_dtype(torch):
    return torch.bfloat16 if QK_TABLE == "bf16" else torch.float32


def build_inputs(torch, binding, inputs, device):
    """All inputs of one step, resident on the device."""
    dt = torch.float16 if ROW_DTYPE == "f16" else torch.bfloat16
    rms = []
    for i, (M, N) in enumerate(RMS_SHAPES):
        x, w = inputs.rmsnorm_inputs(M, N, outlier_frac=0.01, device=device, seed=100 * i,
                                     dtype=dt)
        y = torch.empty_like(x)
        rms.append({"M": M, "N": N, "x": x, "w": w, "y": y})
    for i, (M, N) in enumerate(ADD_SHAPES):
        x, w = inputs.rmsnorm_inputs(M, N, outlier_frac=0.01, device=device, seed=500 + i,
                                     dtype=dt)
        r, _ = inputs.rmsnorm_inputs(M, N, device=device, seed=550 + i, dtype=dt)
        rms.append({"M": M, "N": N, "x": x, "w": w, "y": torch.empty_like(x), "r": r,
                    "h": torch.empty_like(x)})
    for i, (M, N) in enumerate(LN_SHAPES):
        x, w = inputs.rmsnorm_inputs(M, N, outlier_frac=0.01, device=device, seed=700 + i,
                                     dtype=dt)
        rms.append({"M": M, "N": N, "x": x, "w": w, "y": torch.empty_like(x),
                    "b": inputs.norm_bias(N, device=device, seed=750 + i, dtype=dt)})
    for i, (M, N) in enumerate(L2_SHAPES):
        x, _ = inputs.rmsnorm_inputs(M, N, outlier_frac=0.01, device=device, seed=900 + i,
                                     dtype=dt)
        rms.append({"M": M, "N": N, "x": x, "y": torch.empty_like(x), "l2": True})
    qk = []
    for j, r in enumerate(QK_ROT):
        qkv, wq, wk, pos = inputs.qkv_inputs(QK_T, HQ, HKV, D, positions="uniform",
                                             max_pos=MAX_POS, device=device, seed=1000 + j)
        table = binding.rope_cos_sin_table(THETA, MAX_POS, r, device=device, dtype=table_dtype(torch))
        qk.append({"r": r, "qkv": qkv, "wq": wq, "wk": wk, "pos": pos, "table": table})
    return rms, qk


FORCE = {"rms": 0, "qk": 0}  # schedule overrides (--rms-schedule / --qk-schedule)
# The row norms' workspace (dynamic unit order on the row ring): one, shared by
# every row launch, which all run in stream order.  None with --no-workspace.
WS = {"ws": None}


def launch_row(binding, c):
    ws = WS["ws"]
    if "r" in c:
        binding.add_rmsnorm_fwd(c["x"], c["r"], c["w"], RMS_EPS, c["h"], c["y"],
                                schedule=FORCE["rms"], workspace=ws)
    elif "b" in c:
        binding.layernorm_fwd(c["x"], c["w"], c["b"], 1e-5, c["y"], schedule=FORCE["rms"],
                              workspace=ws)
    elif "l2" in c:
        binding.l2norm_fwd(c["x"], 1e-12, c["y"], schedule=FORCE["rms"], workspace=ws)
    else:
        binding.rmsnorm_fwd(c["x"], c["w"], RMS_EPS, c["y"], schedule=FORCE["rms"], workspace=ws)


def launch_qk(binding, c):
    binding.qk_norm_rope_fwd(c["qkv"], c["wq"], c["wk"], c["table"], c["pos"], HQ, HKV, D,
                             c["r"], QK_EPS, schedule=FORCE["qk"])


def launch_step(binding, rms, qk, events=None, skip=None):
    """Enqueue one step; optionally record an event before every launch, or
    leave out launch number `skip`."""
    k = 0
    for c in rms:
        if events is not None:
            events[k].record()
        if k != skip:
            launch_row(binding, c)
        k += 1
    for c in qk:
        if events is not None:
            events[k].record()
        if k != skip:
            launch_qk(binding, c)
        k += 1
    return k


def marginal_ms(torch, binding, rms, qk, n_launch: int, steps: int, rounds: int = 3) -> list:
    """What each launch adds to the step in context: the time of `steps`
    whole steps minus that of the same steps without the launch, both timed
    as pass A times (one event pair, launches overlapping their gaps),
    interleaved, median of `rounds`; milliseconds per step."""
    def timed(skip):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            launch_step(binding, rms, qk, skip=skip)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    out = []
    for i in range(n_launch):
        diffs = [timed(None) - timed(i) for _ in range(rounds)]
        out.append(statistics.median(diffs))
    return out


def graph_ms(torch, launch, reps: int) -> float:
    """Milliseconds per launch of `launch(i)`, i = 0..reps-1, captured once in
    a CUDA graph and replayed: the GPU time of back-to-back launches without
    the host's per-call cost (which exceeds a whole kernel below a few MB)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(4):
            launch(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(reps):
            launch(i)
    graph.replay()
    torch.cuda.synchronize()
    start.record()
    graph.replay()
    end.record()
    torch.cuda.synchronize()
    del graph
    return start.elapsed_time(end) / reps


def direct_ms(torch, launch, reps: int) -> float:
    """Milliseconds per launch issued one by one from Python (host-bound for
    small launches: the figure a caller without graphs sees)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    for i in range(4):
        launch(i)
    torch.cuda.synchronize()
    start.record()
    for i in range(reps):
        launch(i)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / reps


def config_points(torch, binding, inputs, hbm_peak: float) -> dict:
    """The named configurations outside the step, each timed by CUDA-graph
    replay of back-to-back launches on two alternating buffer sets:
    RMSNorm 64 x 4096 (latency), the 32768-wide rows (eps 1e-5), QK at
    T in {1, 2, 16, 64, 256} (rotary 128, positions 0..T-1, latency) and at
    T in {1024, 4096} (rotary 128 and 64, uniform positions)."""
    out = {}

    def rms_point(M, N, eps, latency):
        pair = [inputs.rmsnorm_inputs(M, N, device="cuda", seed=s) for s in (11, 12)]
        ys = [torch.empty_like(pair[0][0]) for _ in range(2)]
        fn = lambda i: binding.rmsnorm_fwd(pair[i & 1][0], pair[0][1], eps, ys[i & 1],  # noqa: E731
                                           workspace=WS["ws"])
        ms = graph_ms(torch, fn, 100 if latency else 20)
        b = rms_bytes(M, N)
        pt = {"M": M, "N": N, "eps": eps, "us": round(ms * 1e3, 2),
              "gbs": round(b / (ms * 1e-3) / 1e9, 1),
              "frac_of_measured": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)}
        if latency:
            pt["us_direct_launch"] = round(direct_ms(torch, fn, 200) * 1e3, 2)
        return pt

    def qk_point(T, r, positions, latency):
        table = binding.rope_cos_sin_table(THETA, MAX_POS, r, device="cuda",
                                           dtype=table_dtype(torch))
        bufs = [inputs.qkv_inputs(T, HQ, HKV, D, positions=positions, max_pos=MAX_POS,
                                  device="cuda", seed=s) for s in (21, 22)]

        def fn(i):
            q, wq, wk, pos = bufs[i & 1]
            binding.qk_norm_rope_fwd(q, wq, wk, table, pos, HQ, HKV, D, r, QK_EPS)

        ms = graph_ms(torch, fn, 100 if latency else 20)
        b = qk_bytes(T, r)
        qs = binding.qk_norm_rope_select_schedule(T, D, r)
        pt = {"T": T, "rotary_dim": r, "positions": positions,
              "kernel": QK_KERNELS.get(qs, str(qs)), "us": round(ms * 1e3, 2),
              "gbs": round(b / (ms * 1e-3) / 1e9, 1),
              "frac_of_measured": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)}
        if latency:
            pt["us_direct_launch"] = round(direct_ms(torch, fn, 200) * 1e3, 2)
        return pt

    out["rmsnorm_64x4096_latency"] = rms_point(64, 4096, 1e-6, True)
    out["rmsnorm_wide_N32768"] = [rms_point(M, 32768, 1e-5, False) for M in (1024, 4096, 8192)]
    out["qk_small_T_latency"] = [qk_point(T, 128, "arange", True) for T in (1, 2, 16, 64, 256)]
    out["qk_T1024_T4096"] = [qk_point(T, r, "uniform", False) for T in (1024, 4096)
                             for r in (128, 64)]
    out["timing"] = ("CUDA-graph replay of back-to-back launches on two alternating buffer "
                     "sets (us per launch); us_direct_launch: the same launches issued one "
                     "by one from Python")
    return out


def steady_per_shape(torch, binding, rms, qk, reps: int, hbm_peak: float) -> list:
    """Each launch of the step measured on its own, in steady state: `reps`
    back-to-back launches of one shape, replayed from a CUDA graph, alternating
    between two sets of activations so nothing is reused from L2 when the
    shape exceeds it (weights and tables shared).
    A launch then pays for the dirty L2 lines its predecessor (the same
    shape) left behind and leaves as many itself, so its DRAM traffic equals
    its algorithmic bytes.  The in-step per-launch times instead also carry
    the dirty tail of whichever launch ran before (up to the 126 MiB L2).
    Beside each: a plain torch streaming kernel over the same number of
    bytes, timed the same way (the ceiling any single-pass kernel of that
    size meets)."""
    out = []

    def copy_frac(nbytes: int) -> float:
        # A plain streaming kernel over the same bytes (half read, half
        # written), run the same way: torch's elementwise bitwise NOT on int32
        # words, the ceiling a single-pass kernel of this size reaches.  (Not
        # copy_: inside a CUDA graph a same-dtype copy becomes a memcpy node
        # whose engine the driver picks, and it measured 2x slower on some
        # buffers.)
        n = nbytes // 2 // 16 * 4
        bufs = [(torch.empty(n, dtype=torch.int32, device="cuda"),
                 torch.empty(n, dtype=torch.int32, device="cuda")) for _ in range(2)]
        ms = timed(bufs, lambda _b, p: torch.bitwise_not(p[0], out=p[1]))
        del bufs
        return round(8 * n / (ms * 1e-3) / 1e9 / hbm_peak, 4)

    def timed(pair, launch):
        return graph_ms(torch, lambda i: launch(binding, pair[i & 1]), reps)

    for c in rms:
        twin = dict(c)
        for k in ("x", "r"):
            if k in c:
                twin[k] = c[k].clone()
        for k in ("y", "h"):
            if k in c:
                twin[k] = torch.empty_like(c[k])
        ms = timed((c, twin), launch_row)
        del twin
        op = ("add_rmsnorm" if "r" in c else "layernorm" if "b" in c else
              "l2norm" if "l2" in c else "rmsnorm")
        b = {"add_rmsnorm": add_bytes, "layernorm": ln_bytes, "l2norm": l2_bytes,
             "rmsnorm": rms_bytes}[op](c["M"], c["N"])
        gbs = b / (ms * 1e-3) / 1e9
        out.append({"op": op, "M": c["M"], "N": c["N"], "us": round(ms * 1e3, 2),
                    "gbs": round(gbs, 1), "frac_of_measured": round(gbs / hbm_peak, 4),
                    "stream_same_bytes_frac": copy_frac(b)})
    for c in qk:
        twin = dict(c)
        twin["qkv"] = c["qkv"].clone()
        ms = timed((c, twin), launch_qk)
        del twin
        b = qk_bytes(QK_T, c["r"])
        gbs = b / (ms * 1e-3) / 1e9
        out.append({"op": "qk_norm_rope", "T": QK_T, "rotary_dim": c["r"],
                    "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                    "frac_of_measured": round(gbs / hbm_peak, 4),
                    "stream_same_bytes_frac": copy_frac(b),
                    "gbs_counting_v": round((b + qk_v_bytes(QK_T)) / (ms * 1e-3) / 1e9, 1)})
    return out


def run_ours(args) -> int:
    import torch

    from row_normalization_gb300 import binding, inputs
    from row_normalization_gb300.build import build

    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    if rank == 0:
        build()
    if dist:
        dist.barrier()
    binding.load()
    device = torch.device("cuda", local)

    rms, qk = build_inputs(torch, binding, inputs, device)
    if not args.no_workspace:
        WS["ws"] = binding.new_workspace(device)
    n_launch = len(rms) + len(qk)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        launch_step(binding, rms, qk)
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start_i = torch.cuda.Event(enable_timing=True)
    end_i = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    # Pass A (the value): K steps exactly as a caller runs them, one event
    # pair around the whole region, so consecutive launches overlap their
    # launch gaps (programmatic dependent launch).
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start.record()
    for s in range(K):
        launch_step(binding, rms, qk)
    end.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    # Pass B (per-launch durations for per_shape and the roofline): the same K
    # steps with an event before every launch.  An event between two kernels
    # serialises them, so these durations carry every launch gap.
    start_i.record()
    for s in range(K):
        launch_step(binding, rms, qk, ev[s])
        ev[s][n_launch].record()
    end_i.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()

    total_ms = start.elapsed_time(end)
    instrumented_ms = start_i.elapsed_time(end_i)
    total_ms = max_over_ranks(torch, dist, total_ms, device)
    per_launch_ms = [statistics.fmean(ev[s][k].elapsed_time(ev[s][k + 1]) for s in range(K))
                     for k in range(n_launch)]

    bytes_step = step_bytes()
    value = job_gbs(world, bytes_step * K, total_ms)
    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    per_shape = []
    for k, c in enumerate(rms):
        op = ("add_rmsnorm" if "r" in c else "layernorm" if "b" in c else
              "l2norm" if "l2" in c else "rmsnorm")
        opcode = {"add_rmsnorm": binding.RN_OP_ADD_RMSNORM, "layernorm": binding.RN_OP_LAYERNORM,
                  "l2norm": binding.RN_OP_L2NORM, "rmsnorm": binding.RN_OP_RMSNORM}[op]
        sched = FORCE["rms"] or binding.row_norm_select_schedule(
            opcode, c["M"], c["N"], workspace=WS["ws"] is not None)
        b = {"add_rmsnorm": add_bytes, "layernorm": ln_bytes, "l2norm": l2_bytes,
             "rmsnorm": rms_bytes}[op](c["M"], c["N"])
        per_shape.append({"op": op, "dtype": ROW_DTYPE, "M": c["M"], "N": c["N"],
                          "kernel": RMS_KERNELS.get(sched, str(sched)),
                          "us": round(per_launch_ms[k] * 1e3, 2), "bytes": b,
                          "gbs": round(b / (per_launch_ms[k] * 1e-3) / 1e9, 1)})
    for j, c in enumerate(qk):
        k = len(rms) + j
        b = qk_bytes(QK_T, c["r"])
        qs = FORCE["qk"] or binding.qk_norm_rope_select_schedule(QK_T, D, c["r"])
        per_shape.append({"op": "qk_norm_rope", "T": QK_T, "rotary_dim": c["r"],
                          "kernel": QK_KERNELS.get(qs, str(qs)),
                          "us": round(per_launch_ms[k] * 1e3, 2), "bytes": b,
                          "gbs": round(b / (per_launch_ms[k] * 1e-3) / 1e9, 1),
                          "gbs_counting_v": round((b + qk_v_bytes(QK_T))
                                                  / (per_launch_ms[k] * 1e-3) / 1e9, 1)})
    marg = marginal_ms(torch, binding, rms, qk, n_launch, args.marginal_steps) \
        if args.marginal_steps > 0 else None
    for k, p in enumerate(per_shape):
        p["frac_of_measured"] = round(p["gbs"] / hbm_peak, 4)
        if marg is not None and marg[k] > 0:
            p["marginal_us"] = round(marg[k] * 1e3, 2)
            p["marginal_frac_of_measured"] = round(p["bytes"] / (marg[k] * 1e-3) / 1e9 / hbm_peak, 4)
        wl = (f"{p['op']} M={p['M']} N={p['N']}" if p["op"] != "qk_norm_rope"
              else f"qk_norm_rope T={p['T']} r={p['rotary_dim']}")
        p["ncu"] = ncu_counters(p["kernel"], wl)
    dom = max(per_shape, key=lambda p: p["us"])
    dom_wl = (f"{dom['op']} M={dom['M']} N={dom['N']}" if dom["op"] != "qk_norm_rope"
              else f"qk_norm_rope T={dom['T']} r={dom['rotary_dim']}")
    achieved = dom["bytes"] / (dom["us"] * 1e-6) / 1e9
    dom_ncu = ncu_counters(dom["kernel"], dom_wl)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                "traffic": (dom_ncu["dram_bytes_read"] + dom_ncu["dram_bytes_write"]
                            if dom_ncu else None),
                "dram_bytes_read": dom_ncu["dram_bytes_read"] if dom_ncu else None,
                "dram_bytes_write": dom_ncu["dram_bytes_write"] if dom_ncu else None,
                "dram_throughput_pct_of_peak": (dom_ncu["dram_throughput_pct_of_peak"]
                                                if dom_ncu else None),
                "kernel": dom["kernel"], "launch": dom_wl,
                "algorithmic_bytes_per_launch": dom["bytes"]}

    steady = steady_per_shape(torch, binding, rms, qk, args.steady_reps, hbm_peak) \
        if args.steady_reps > 0 else None
    plain = not ADD_SHAPES and not LN_SHAPES and not L2_SHAPES and ROW_DTYPE == "bf16"
    configs = config_points(torch, binding, inputs, hbm_peak) \
        if plain and WORKLOAD.startswith("rmsnorm sweep") and args.steady_reps > 0 else None
    e2e = run_e2e(torch, binding, rms, qk, args, dist, device) if args.e2e_steps > 0 and plain \
        else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and plain:
        cpu = cpu_baseline(budget_s=args.cpu_seconds)

    rms_ms = sum(per_launch_ms[:len(RMS_SHAPES)])
    qk_ms = sum(per_launch_ms[len(rms):])
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
        "ms_per_step_with_per_launch_events": round(instrumented_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (ROW_DTYPE if ROW_DTYPE == "bf16" or not QK_ROT
                  else f"{ROW_DTYPE} (row norms), bf16 (qk_norm_rope)"),
        "data": "synthetic (seeded torch generators: x ~ N(0,1) with 1% outlier rows x100, w = 1 + 0.1 N(0,1); QKV ~ N(0,1), positions uniform)",
        "config": {"workload": WORKLOAD, "bytes_per_step": bytes_step,
                   "launches_per_step": n_launch, "parallelism": f"replicas x{world}",
                   "row_entry": ("rmsnorm_fwd_ws: one caller-owned workspace, dynamic unit order "
                                 "on the row ring" if WS["ws"] is not None else
                                 "rmsnorm_fwd: fixed unit order"),
                   "qk_cos_sin_table": "bf16" if QK_TABLE == "bf16" else "fp32",
                   "l2": (("inputs larger than L2: each buffer is touched once per step and a "
                           f"step moves {bytes_step / 1e9:.2f} GB, "
                           f"{bytes_step / L2_BYTES:.0f}x the 126 MiB L2")
                          if bytes_step >= 4 * L2_BYTES else
                          (f"step of {bytes_step / 1e9:.2f} GB is under 4x the 126 MiB L2: "
                           "in-step numbers may reuse L2; steady_per_shape alternates two "
                           "buffer sets"))},
        "frac_of_measured_copy": round(value / world / hbm_peak, 4),
        "frac_of_spec_7928": round(value / world / SPEC_GBS, 4),
        "per_op": {"rmsnorm_sweep_gbs": round(sum(rms_bytes(M, N) for M, N in RMS_SHAPES)
                                              / (rms_ms * 1e-3) / 1e9, 1) if rms_ms else None,
                   "qk_norm_rope_gbs": round(sum(qk_bytes(QK_T, r) for r in QK_ROT)
                                             / (qk_ms * 1e-3) / 1e9, 1) if qk_ms else None},
        "timing": ("value and ms_per_step: K steps with one event pair around them "
                   "(launches overlap their gaps through programmatic dependent launch); "
                   "per_shape and roofline: a second pass of the same K steps with an event "
                   "before every launch, which serialises the launches; per_shape marginal_us: "
                   "the step's time minus that of the step without the launch, both timed "
                   "like the value (what the launch costs in context)"),
        "per_shape": per_shape,
        "steady_per_shape": steady,
        "configs": configs,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_launch * K,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


E2E_CHUNK_BYTES = 64 << 20


def link_copy_gbs(torch, device, nbytes: int = 512 << 20, reps: int = 5, streams=None) -> float:
    """What this host link carries with both directions busy: one pinned
    host-to-device and one device-to-host copy of `nbytes` each, on two
    streams at once, median of `reps` (GB/s, both directions added up).  The
    e2e pipeline moves the same two directions, so its `link_gbs` is read
    against this."""
    hin = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    hout = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dout = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = streams or (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    times = []
    for _ in range(reps + 1):
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s1):
            din.copy_(hin, non_blocking=True)
        with torch.cuda.stream(s2):
            hout.copy_(dout, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s1)
        torch.cuda.current_stream().wait_stream(s2)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times[1:])
    del hin, hout, din, dout
    return 2 * nbytes / (ms * 1e-3) / 1e9


def run_e2e(torch, binding, rms, qk, args, dist, device, streams=None):
    """The same step with host buffers, through the same C entry points.

    Every step copies each activation (x, qkv, positions) in from pinned host
    memory and each result (y, qkv) back, inside the timed region.  The work
    is cut into ~64 MB chunks and pipelined over three streams -- host-to-
    device copies, kernels, device-to-host copies -- ordered by events, so the
    two copy directions and the kernels overlap.  Weights and the cos/sin
    table stay resident."""
    world = dist.get_world_size() if dist else 1
    s_in, s_comp, s_out = streams or tuple(torch.cuda.Stream(device=device) for _ in range(3))

    # one entry per chunk: (kind, device views, pinned host views, launch args)
    chunks = []
    for c in rms:
        xh = c["x"].cpu().pin_memory()
        yh = torch.empty_like(c["y"], device="cpu").pin_memory()
        rows = max(1, E2E_CHUNK_BYTES // (c["N"] * 2))
        for r0 in range(0, c["M"], rows):
            r1 = min(c["M"], r0 + rows)
            chunks.append(("rms", c, (c["x"][r0:r1], c["y"][r0:r1]), (xh[r0:r1], yh[r0:r1])))
    for c in qk:
        qh = c["qkv"].cpu().pin_memory()
        ph = c["pos"].cpu().pin_memory()
        oh = torch.empty_like(c["qkv"], device="cpu").pin_memory()
        toks = max(1, E2E_CHUNK_BYTES // (c["qkv"].shape[1] * 2))
        for t0 in range(0, QK_T, toks):
            t1 = min(QK_T, t0 + toks)
            chunks.append(("qk", c, (c["qkv"][t0:t1], c["pos"][t0:t1]),
                           (qh[t0:t1], ph[t0:t1], oh[t0:t1])))
    h2d = sum(h[0].numel() * h[0].element_size() + (h[1].numel() * 8 if k == "qk" else 0)
              for k, _, _, h in chunks)
    d2h = sum((h[1] if k == "rms" else h[2]).numel() * 2 for k, _, _, h in chunks)

    link_peak = link_copy_gbs(torch, device, streams=(s_in, s_out))

    n = len(chunks)
    done_comp = [None] * n  # kernel of the previous step on this chunk (WAR for the copy in)
    done_out = [None] * n   # copy-out of the previous step (WAR for the kernel's output)

    def one_step():
        for i, (kind, c, dv, hv) in enumerate(chunks):
            with torch.cuda.stream(s_in):
                if done_comp[i] is not None:
                    s_in.wait_event(done_comp[i])
                dv[0].copy_(hv[0], non_blocking=True)
                if kind == "qk":
                    dv[1].copy_(hv[1], non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            s_comp.wait_event(e_in)
            if done_out[i] is not None:
                s_comp.wait_event(done_out[i])
            if kind == "rms":
                binding.rmsnorm_fwd(dv[0], c["w"], RMS_EPS, dv[1], stream=s_comp,
                                    workspace=WS["ws"])
                out_dev, out_host = dv[1], hv[1]
            else:
                binding.qk_norm_rope_fwd(dv[0], c["wq"], c["wk"], c["table"], dv[1], HQ, HKV, D,
                                         c["r"], QK_EPS, stream=s_comp)
                out_dev, out_host = dv[0], hv[2]
            e_c = torch.cuda.Event()
            e_c.record(s_comp)
            done_comp[i] = e_c
            s_out.wait_event(e_c)
            with torch.cuda.stream(s_out):
                out_host.copy_(out_dev, non_blocking=True)
                e_o = torch.cuda.Event()
                e_o.record(s_out)
            done_out[i] = e_o

    for _ in range(2):
        one_step()
    torch.cuda.synchronize()
    E = args.e2e_steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(s_in)
    s_comp.wait_event(start)
    s_out.wait_event(start)
    for _ in range(E):
        one_step()
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3
    ms = start.elapsed_time(end)
    ms = max_over_ranks(torch, dist, ms, device)
    val = job_gbs(world, step_bytes() * E, ms)
    return {"value": round(val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": round(ms / E, 3),
            "host_wall_ms_per_step": round(wall_ms / E, 3),
            "link_gbs": round((h2d + d2h) / (ms / E * 1e-3) / 1e9, 1),
            "link_peak_gbs": round(link_peak, 1),
            "link_frac": round((h2d + d2h) / (ms / E * 1e-3) / 1e9 / link_peak, 4),
            "note": ("activations in from pinned host memory and results back every step, "
                     f"{n} chunks of <= 64 MB pipelined over copy-in / kernel / copy-out streams; "
                     "weights and the cos/sin table stay resident")}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and the reference arm)
# ---------------------------------------------------------------------------

def _cpu_sample(frac_den: int):
    """A bounded sample of the workload on the host: the first ceil(M/frac_den)
    rows of every RMSNorm shape and the first ceil(T/frac_den) tokens of each
    QK case, with inputs drawn by the same generators (host device)."""
    import numpy as np

    import oracle
    from row_normalization_gb300.inputs import bf16_bits, qkv_inputs, rmsnorm_inputs
    rms = []
    for i, (M, N) in enumerate(RMS_SHAPES):
        m = max(1, math.ceil(M / frac_den))
        x, w = rmsnorm_inputs(m, N, outlier_frac=0.01, device="cpu", seed=100 * i)
        rms.append((bf16_bits(x), bf16_bits(w)))
    qk = []
    for j, r in enumerate(QK_ROT):
        t = max(1, math.ceil(QK_T / frac_den))
        qkv, wq, wk, pos = qkv_inputs(t, HQ, HKV, D, positions="uniform", max_pos=MAX_POS,
                                      device="cpu", seed=1000 + j)
        qk.append((bf16_bits(qkv), bf16_bits(wq), bf16_bits(wk), pos.numpy(), r))
    if QK_TABLE == "bf16":  # the oracle reads bf16 entries widened exactly to fp32
        tables = {r: (oracle.rope_cos_sin_bf16(THETA, MAX_POS, r).astype(np.uint32) << 16)
                  .view(np.float32) for r in QK_ROT}
    else:
        tables = {r: oracle.rope_cos_sin(THETA, MAX_POS, r) for r in QK_ROT}
    nbytes = sum(rms_bytes(x.shape[0], x.shape[1]) for x, _ in rms) + \
        sum(qk_bytes(q[0].shape[0], q[4]) for q in qk)
    return rms, qk, tables, nbytes, np


def _cpu_pass(pool, threads, rms, qk, tables):
    import numpy as np

    import oracle
    futs = []
    for x, w in rms:
        for part in np.array_split(np.arange(x.shape[0]), min(threads, x.shape[0])):
            if part.size:
                futs.append(pool.submit(oracle.rmsnorm, x[part[0]:part[-1] + 1], w, RMS_EPS))
    for qkv, wq, wk, pos, r in qk:
        for part in np.array_split(np.arange(qkv.shape[0]), min(threads, qkv.shape[0])):
            if part.size:
                a, b = part[0], part[-1] + 1
                futs.append(pool.submit(oracle.qk_norm_rope, qkv[a:b], wq, wk, tables[r],
                                        pos[a:b], HQ, HKV, D, r, QK_EPS))
    for f in futs:
        f.result()


def cpu_baseline(budget_s: float = 10.0, frac_den: int = 256) -> dict:
    """Times the oracle, unchanged, on the host cores: rows and tokens are split
    over one thread per core (the C oracle releases the GIL), and whole passes
    over the sample repeat until about `budget_s` seconds have run."""
    threads = len(os.sched_getaffinity(0))
    rms, qk, tables, nbytes, _ = _cpu_sample(frac_den)
    passes = 0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        while True:
            _cpu_pass(pool, threads, rms, qk, tables)
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    # one thread on the same sample, for a fraction of the budget
    single = None
    with ThreadPoolExecutor(max_workers=1) as pool1:
        t1 = time.perf_counter()
        p1 = 0
        while True:
            _cpu_pass(pool1, 1, rms, qk, tables)
            p1 += 1
            e1 = time.perf_counter() - t1
            if e1 >= budget_s * 0.3:
                break
        single = round(nbytes * p1 / e1 / 1e9, 3)
    return {"value": round(nbytes * passes / el / 1e9, 3), "unit": "GB/s", "cores": threads,
            "single_thread_value": single, "kind": "oracle",
            "sample": (f"first 1/{frac_den} of the rows of every RMSNorm shape and of the "
                       f"tokens of each QK case ({nbytes / 1e6:.1f} MB ideal traffic per pass), "
                       f"{passes} passes in {el:.1f} s, fp64 C oracle on {threads} threads")}


def run_reference(args) -> int:
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    threads = len(os.sched_getaffinity(0))
    # size each step so the whole run stays near a minute and a half
    budget = 90.0 / max(1, args.steps + args.warmup)
    frac_den = 256
    rms, qk, tables, nbytes, _ = _cpu_sample(frac_den)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        _cpu_pass(pool, threads, rms, qk, tables)
        one = time.perf_counter() - t0
        scale = max(1, int(round(one / budget)))
        if scale > 1:
            frac_den *= scale
            rms, qk, tables, nbytes, _ = _cpu_sample(frac_den)
        for _ in range(args.warmup):
            _cpu_pass(pool, threads, rms, qk, tables)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            _cpu_pass(pool, threads, rms, qk, tables)
        el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    sample = (f"each step: first 1/{frac_den} of the rows of every RMSNorm shape and of the "
              f"tokens of each QK case ({nbytes / 1e6:.2f} MB ideal traffic)")
    line = {"metric": METRIC, "impl": "reference", "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample,
                       "qk_cos_sin_table": "bf16" if QK_TABLE == "bf16" else "fp32"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--marginal-steps", type=int, default=200,
                    help="steps per timing of each launch's marginal cost in the step (0: skip)")
    ap.add_argument("--steady-reps", type=int, default=50,
                    help="back-to-back launches per shape for steady_per_shape (0: skip)")
    ap.add_argument("--only", default="", help="profile a subset, e.g. rms:8192x16384")
    ap.add_argument("--qk-table", choices=("f32", "bf16"), default="f32",
                    help="element type of the rotary cos/sin table the QK launches read")
    ap.add_argument("--row-dtype", choices=("bf16", "f16"), default="bf16",
                    help="element format of the row norms in the step (the QK op stays bf16)")
    ap.add_argument("--rms-schedule", type=int, default=0, help="force an RN_SCHED_* value")
    ap.add_argument("--no-workspace", action="store_true",
                    help="row norms without a workspace (the ring's fixed unit order)")
    ap.add_argument("--qk-schedule", type=int, default=0, help="force an RN_QK_* value")
    args = ap.parse_args()
    FORCE["rms"], FORCE["qk"] = args.rms_schedule, args.qk_schedule
    if args.only:
        restrict_workload(args.only)
    global ROW_DTYPE, QK_TABLE
    ROW_DTYPE = args.row_dtype
    QK_TABLE = args.qk_table
    if args.impl == "ours" and args.warmup < 3:
        args.warmup = 3  # never time without at least three warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
