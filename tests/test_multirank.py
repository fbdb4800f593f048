"""The bench's multi-rank logic on CPU: two gloo ranks, 127.0.0.1 rendezvous.

Each rank decodes its own batch (weak scaling, no collective on the data path); the
only collectives are the timing reductions: the max of the ranks' times and the
sum of their step counts.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, lr, w = bench.dist_env()
        times = [3.5, 1.25]
        steps = [10, 20]
        out[rank] = (r, lr, w, bench.max_over_ranks(times[rank], w), bench.sum_over_ranks(steps[rank], w),
                     bench.rank_seed(1236, r))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_times_and_counts():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        rank, local, world, tmax, ssum, seed = res[r]
        assert (rank, local, world) == (r, r, 2)
        assert tmax == 3.5                      # the slowest rank sets the time
        assert ssum == 30                       # whole-job units
    assert res[0][5] != res[1][5]               # distinct inputs per rank


def test_single_process_defaults(monkeypatch):
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(2.0, 1) == 2.0 and bench.sum_over_ranks(5, 1) == 5


def _gather_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import verify_bs_step_gb300 as vbs
        part = torch.full((40,), rank + 1, dtype=torch.uint8)
        part[0] = 200 + rank
        got = vbs.gather_shard_partials(part)
        out[rank] = got.tolist()
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_vocab_shard_partials_gather_in_rank_order():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in (0, 1):
        rows = res[r]
        assert len(rows) == 2
        for k in (0, 1):
            assert rows[k][0] == 200 + k and rows[k][1:] == [k + 1] * 39


def test_oracle_all_cores_sums_the_processes():
    """The all-core cpu_baseline: spawned processes, each timing its own sentence after a
    common start; the units add up and the time is the longest process's."""
    import bench
    units, el, n = bench.oracle_all_cores(0.3, n=2)
    assert n == 2 and units >= 2 and el >= 0.3
