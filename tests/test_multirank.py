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


def _bench(args, env_extra=None, timeout=300):
    import json
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    env.update(env_extra or {})
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
                         capture_output=True, text=True, timeout=timeout)
    lines = [json.loads(l) for l in out.stdout.splitlines() if l.startswith("{")]
    return out.returncode, lines, out.stderr


def test_bench_gpus_flag_starts_its_own_ranks():
    """`bench.py --gpus 2` with no launcher around it starts two ranks itself
    (gloo here, no GPU): rank 0 prints one line with both ranks' seeds and the
    max-over-ranks timings."""
    rc, lines, err = _bench(["--gpus", "2", "--launcher-check"])
    assert rc == 0, err[-2000:]
    assert len(lines) == 1, lines
    d = lines[0]
    assert d["n_ranks"] == 2 and d["gpus_flag"] == 2
    assert d["seeds"] == [[1, 4], [1001, 1004]]
    assert d["max_over_ranks"] == [2.0, 4.0]


def test_bench_refuses_more_gpus_than_visible():
    rc, lines, err = _bench(["--gpus", "2", "--steps", "1"])
    assert rc == 2 and not lines
    assert "GPU(s) visible" in err


def test_bench_refuses_world_size_mismatch():
    rc, lines, err = _bench(["--gpus", "4", "--launcher-check"], {"WORLD_SIZE": "2", "RANK": "0"})
    assert rc == 2 and not lines
    assert "WORLD_SIZE" in err
