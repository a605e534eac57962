"""The bench's multi-process host logic on CPU (gloo, world size 2).

The path is replicas only: every rank runs the whole step on its own GPU and
the ranks share no data.  What the ranks do share is host logic: the slowest
rank's time, the whole-job value over all ranks, and the reference arm that
only rank 0 runs.  No GPU is involved here.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is slower
        slowest = bench.max_over_ranks(torch, dist, mine, torch.device("cpu"))
        out.put((rank, slowest, bench.job_gbs(world, 7_000_000_000, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]
    # both ranks moved 7 GB in the slowest rank's 15 ms: 2 x 7e9 B / 15e-3 s
    assert all(abs(g[2] - 2 * 7e9 / 15e-3 / 1e9) < 1e-6 for g in got)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(torch, None, 12.5, torch.device("cpu")) == 12.5
    assert bench.job_gbs(1, 2_000_000_000, 1000.0) == 2.0


def test_reference_arm_runs_on_rank_zero_only():
    # under torchrun every rank starts the reference arm; ranks other than 0
    # leave at once with status 0 and print nothing
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    # rank 0 of the reference arm: one JSON line with the contract's keys, the
    # oracle timed on the host cores, and an e2e that copies nothing
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1"], env=env, capture_output=True,
                         text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
