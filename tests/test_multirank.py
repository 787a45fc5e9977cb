"""Host-side logic of the multi-GPU bench path, run as two gloo ranks on CPU.

With N GPUs every rank runs the same step on its own GPU with its own seeds
(independent problems; no collective on the data path); only the timing
needs a collective: the job's time is the maximum over ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], dist)
        wp, wd = bench.rank_workloads(rank)
        out[rank] = (got, wp.seed, wd.seed, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_times_and_split_seeds():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        got, sp, sd, env = res[r]
        assert got == [2.0, 10.0, 0.5]          # max over ranks, on every rank
        assert env == (r, world, 0)
    # independent problems: each rank draws different inputs
    assert res[0][1] != res[1][1] and res[0][2] != res[1][2]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.0], None) == [3.0, 4.0]
