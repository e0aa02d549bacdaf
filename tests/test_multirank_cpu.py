"""The data-parallel sharding of the path, on CPU with two gloo ranks.

The hot path shards over tokens with no exchange: every rank quantises and
multiplies its own rows with the same (replicated) weight.  Each rank here
computes its row shard with the oracle; the gathered shards must equal the
unsharded computation bit for bit, and the max-over-ranks timing reduction
used by the benchmark must return the slowest rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    from fp8_fine_grained_fp8bs_gb300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, w = synth.tiny_fprop(0)
        rows = np.array_split(np.arange(x.shape[0]), world)[rank]
        qa, sa = oracle.quantize_act_1x128(x[rows])
        qb, sb = oracle.quantize_weight_128x128(w)
        y, _ = oracle.gemm_block_scaled(qa, sa, qb, sb)
        parts = [None] * world
        dist.all_gather_object(parts, (rows, qa, sa, y))
        # slowest-rank timing, as bench.py reduces it
        t = torch.tensor([1.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            q.put((parts, float(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_rank_row_shards_equal_unsharded():
    import oracle
    from fp8_fine_grained_fp8bs_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert tmax == 2.0
    x, w = synth.tiny_fprop(0)
    qa, sa = oracle.quantize_act_1x128(x)
    qb, sb = oracle.quantize_weight_128x128(w)
    y, _ = oracle.gemm_block_scaled(qa, sa, qb, sb)
    rows = np.concatenate([p[0] for p in parts])
    assert np.array_equal(rows, np.arange(x.shape[0]))
    assert np.array_equal(np.concatenate([p[1] for p in parts]), qa)
    assert np.array_equal(np.concatenate([p[2] for p in parts]), sa)
    assert np.array_equal(np.concatenate([p[3] for p in parts]), y)
