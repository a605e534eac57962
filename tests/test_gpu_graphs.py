"""The library under CUDA graph capture (GPU).

Every entry point enqueues stream-ordered launches (programmatic dependent
launch) and allocates nothing, so a CUDA graph can record a whole sequence
of them: a decode loop replays it without the host's per-call cost.  The
graph is captured once over static buffers, then replayed on fresh seeded
data each time; every replay must match the oracle like a direct call.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from row_normalization_gb300 import binding
from row_normalization_gb300.inputs import bf16_bits, norm_bias, qkv_inputs, rmsnorm_inputs
from tests.exact import ulp_distance_bf16
from tests.gpu_util import oracle_table, require_gpu
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_graph_replay_matches_the_oracle_every_op():
    M, N, T, HQ, HKV, D, R = 2000, 4096, 777, 8, 2, 128, 128
    eps = 1e-6
    dev = "cuda"
    x = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    r = torch.empty_like(x)
    x16 = torch.empty(M, N, dtype=torch.float16, device=dev)
    w = rmsnorm_inputs(1, N, seed=3)[1].to(dev)
    w16 = w.float().to(torch.float16)
    b = norm_bias(N, seed=4).to(dev)
    ys = [torch.empty_like(x) for _ in range(4)]
    h = torch.empty_like(x)
    y16 = torch.empty_like(x16)
    qkv = torch.empty(T, (HQ + 2 * HKV) * D, dtype=torch.bfloat16, device=dev)
    _, wq, wk, _ = qkv_inputs(1, HQ, HKV, D, seed=5)
    wq, wk = wq.to(dev), wk.to(dev)
    pos = torch.empty(T, dtype=torch.int64, device=dev)
    table = torch.from_numpy(oracle_table(1e6, 4096, R)).to(dev)
    qkv2 = torch.empty_like(qkv)
    table16 = torch.empty(4096, R, dtype=torch.bfloat16, device=dev)  # built inside the graph

    def step():
        binding.rmsnorm_fwd(x, w, eps, ys[0])
        binding.add_rmsnorm_fwd(x, r, w, eps, h, ys[1])
        binding.layernorm_fwd(x, w, b, 1e-5, ys[2])
        binding.l2norm_fwd(x, 1e-12, ys[3])
        binding.rmsnorm_fwd(x16, w16, eps, y16)
        binding.qk_norm_rope_fwd(qkv, wq, wk, table, pos, HQ, HKV, D, R, eps)
        binding.rope_cos_sin_table(1e6, 4096, R, table16)
        binding.qk_norm_rope_fwd_ex(qkv2, wq, wk, table16, pos, HQ, HKV, D, R, eps,
                                    rope_style=binding.RN_ROPE_GPTJ)

    def fill(seed):
        xs, _ = rmsnorm_inputs(M, N, outlier_frac=0.01, seed=seed)
        rs, _ = rmsnorm_inputs(M, N, seed=seed + 1)
        q, _, _, p = qkv_inputs(T, HQ, HKV, D, positions="uniform", max_pos=4096, seed=seed + 2)
        x.copy_(xs)
        r.copy_(rs)
        x16.copy_(xs.float().to(torch.float16))
        qkv.copy_(q)
        qkv2.copy_(q)
        pos.copy_(p)
        return xs, rs, q, p

    fill(100)  # capture runs on real data once, to warm every path
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (11, 23, 37):
        xs, rs, q, p = fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        xb, rb, wb = bf16_bits(xs), bf16_bits(rs), bf16_bits(w)
        assert_parity(bf16_bits(ys[0]), oracle.rmsnorm(xb, wb, eps), f"graph rmsnorm {seed}")
        h_want, y_want = oracle.add_rmsnorm(xb, rb, wb, eps)
        assert np.array_equal(bf16_bits(h), h_want)
        assert_parity(bf16_bits(ys[1]), y_want, f"graph add {seed}")
        assert_parity(bf16_bits(ys[2]), oracle.layernorm(xb, wb, bf16_bits(b), 1e-5),
                      f"graph layernorm {seed}")
        assert_parity(bf16_bits(ys[3]), oracle.l2norm(xb, 1e-12), f"graph l2norm {seed}")
        x16b = bf16_bits(xs.float().to(torch.float16))
        assert_parity(bf16_bits(y16), oracle.rmsnorm(x16b, bf16_bits(w16), eps, f16=True),
                      f"graph rmsnorm fp16 {seed}", fmt="f16")
        want_q = oracle.qk_norm_rope(bf16_bits(q), bf16_bits(wq), bf16_bits(wk),
                                     oracle_table(1e6, 4096, R), p.numpy(), HQ, HKV, D, R, eps)
        assert_parity(bf16_bits(qkv), want_q, f"graph qk {seed}")
        # the bf16 table the graph builds, then GPT-J pairs reading it
        t16 = bf16_bits(table16)
        assert ulp_distance_bf16(t16, oracle.rope_cos_sin_bf16(1e6, 4096, R)).max() <= 1
        wide = (t16.astype(np.uint32) << 16).view(np.float32)
        want_j = oracle.qk_norm_rope(bf16_bits(q), bf16_bits(wq), bf16_bits(wk), wide, p.numpy(),
                                     HQ, HKV, D, R, eps, style=1)
        assert_parity(bf16_bits(qkv2), want_j, f"graph qk bf16 table gptj {seed}")
