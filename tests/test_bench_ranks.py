"""The bench's multi-rank path (independent replicas, max-over-ranks timing,
whole-job rate) on world_size-2 gloo process groups on the CPU.  The path
has no data exchange between ranks; only the timing reduction crosses them."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from tree_speculative_decoding_jt_gb300 import workloads as wk


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (r + 1) ms per step and an attention time of 5 - r
        got = bench.max_over_ranks([rank + 1.0, 5.0 - rank], "cpu", world)
        rate = bench.whole_job_rate(256, got[0] * 1e-3, world)
        q.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_on_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in out:
        assert got == [2.0, 5.0]                       # slowest rank's step and attention time
        assert rate == pytest.approx(2 * 256 / 2e-3)   # units of both ranks / slowest time


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], "cpu", 1) == [1.5, 2.5]
    assert bench.whole_job_rate(256, 1e-4, 1) == pytest.approx(2.56e6)


def test_replicas_draw_distinct_batches_and_rank0_keeps_the_default():
    cfg = 1
    assert bench.replica_seed(cfg, 0) == 1000 + cfg      # the workload's default seed
    a = wk.make(cfg, seed=bench.replica_seed(cfg, 0))
    b = wk.make(cfg, seed=bench.replica_seed(cfg, 1))
    d = wk.make(cfg)
    np.testing.assert_array_equal(a.q, d.q)
    assert not np.array_equal(a.q, b.q)
    assert a.total == b.total                           # same shapes: weak scaling
