"""Two-rank (gloo, CPU) checks of the host logic bench.py uses for N > 1."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_speculative_gb300 import replicas, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ctx, ql, *_ = synth.config_lengths("mixed_fp8")
        cl, qq, idx = replicas.sub_batch(ctx, ql, world, rank)
        # every rank reports its shard; rank 0 checks the union is the batch, disjointly
        gathered = [None] * world
        dist.all_gather_object(gathered, idx.tolist())
        my_ms = 10.0 + rank  # rank 1 is the slow one
        mx = replicas.max_over_ranks(my_ms)
        tot = replicas.sum_over_ranks(1.0)
        q.put((rank, gathered, mx, tot, sum(cl)))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_and_timing():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    gathered = res[0][1]
    flat = sorted(i for part in gathered for i in part)
    assert flat == list(range(64))
    assert not set(gathered[0]) & set(gathered[1])
    for r in res:
        assert r[2] == 11.0  # max over ranks
        assert r[3] == 2.0
    ctx_all, *_ = synth.config_lengths("mixed_fp8")
    assert res[0][4] + res[1][4] == sum(ctx_all)


def test_job_throughput_is_all_bytes_over_slowest_rank():
    assert replicas.job_throughput(2e9, 10, 1000.0) == pytest.approx(20.0)


def test_single_process_reductions_are_identity():
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.sum_over_ranks(2.0) == 2.0
