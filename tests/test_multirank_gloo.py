"""The multi-rank path on CPU: world size 2 over gloo.

The hot path shards by token rows with no exchange (the sequence-parallelism
post: RMSNorm and the residual add need only the local tokens; RoPE and GEGLU
are per token too).  Each rank computes its row shard with the oracle; the
gathered shards must equal the single-rank result bit for bit.  The bench's
timing aggregation (max over ranks, whole-job throughput) runs through the
same process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from diffusion_transformer_elementwise_rotate_b300 import workloads as W

EPS = float(np.float32(1e-6))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        wl = W.WORKLOADS["tiny"]
        bits = oracle.bf16_bits
        x, r, w = (bits(t) for t in W.rmsnorm_inputs(wl))
        lo, hi = W.shard_rows(wl.T_norm, rank, world)
        h, y = oracle.rmsnorm_residual(x[lo:hi], r[lo:hi], w, EPS)
        gu = bits(W.geglu_inputs(wl))
        glo, ghi = W.shard_rows(wl.T_ff, rank, world)
        g = oracle.gelu_and_mul_fused(gu[glo:ghi])
        q = bits(W.rope_inputs(wl, "q"))
        c, s = oracle.rope_cos_sin(W.freqs_for(wl).numpy())
        tlo, thi = W.shard_rows(wl.S, rank, world)
        o = oracle.rope_rotate_half(q[:, tlo:thi], c[tlo:thi], s[tlo:thi])
        parts = [None] * world
        dist.all_gather_object(parts, (h, y, g, o))
        elapsed = bench.max_over_ranks(10.0 + rank, dist)
        gbs = bench.aggregate_gbs(1_000_000, world, 4, elapsed)
        if rank == 0:
            result_q.put((parts, elapsed, gbs))
    finally:
        dist.destroy_process_group()


def test_shard_rows_partition():
    for n in (0, 1, 7, 256, 32760):
        for world in (1, 2, 3, 8):
            spans = [W.shard_rows(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        W.shard_rows(10, 2, 2)


def test_two_gloo_ranks_shard_tokens_without_exchange():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts, elapsed, gbs = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = W.WORKLOADS["tiny"]
    bits = oracle.bf16_bits
    x, r, w = (bits(t) for t in W.rmsnorm_inputs(wl))
    h_full, y_full = oracle.rmsnorm_residual(x, r, w, EPS)
    assert np.array_equal(np.concatenate([p[0] for p in parts]), h_full)
    assert np.array_equal(np.concatenate([p[1] for p in parts]), y_full)
    g_full = oracle.gelu_and_mul_fused(bits(W.geglu_inputs(wl)))
    assert np.array_equal(np.concatenate([p[2] for p in parts]), g_full)
    c, s = oracle.rope_cos_sin(W.freqs_for(wl).numpy())
    o_full = oracle.rope_rotate_half(bits(W.rope_inputs(wl, "q")), c, s)
    assert np.array_equal(np.concatenate([p[3] for p in parts], axis=1), o_full)
    # max over ranks, and whole-job throughput from it
    assert elapsed == 11.0
    assert abs(gbs - 1_000_000 * 2 * 4 / 0.011 / 1e9) < 1e-12
