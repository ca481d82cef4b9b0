"""Host side of the multi-GPU benchmark path on CPU ranks (gloo, world size 2).

The path shards into independent (b, h_kv) groups, so N GPUs run N
independent batches (weak scaling) and the only collective is the timing
reduction: the job takes as long as its slowest rank.
"""

import os
import socket

import numpy as np
import pytest

import synthetic_inputs as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        q.put((rank, bench.max_over_ranks(1.5 + rank, dist, "cpu")))
    finally:
        dist.destroy_process_group()


def test_timing_is_the_max_over_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=1, impl="reference")
    assert bench.reference_arm(args) == 0
    assert capsys.readouterr().out == ""


def test_ranks_draw_independent_batches():
    # Each rank's bench offsets the workload seed by 1000 x rank.
    wl = S.WORKLOADS["decode_4k"]
    a = S.make_inputs(wl)
    b = S.make_inputs(wl.scaled(seed=wl.seed + 1000))
    assert a.q.shape == b.q.shape and not np.array_equal(a.q, b.q)
