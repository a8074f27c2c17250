"""bench.py's multi-process path (process-group set-up, barrier, max over ranks) with two gloo
ranks on the CPU, launched the way torchrun launches it (RANK / WORLD_SIZE / MASTER_* in the
environment)."""
import argparse
import os

import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import bench

    args = argparse.Namespace(impl="ours")
    w, r, local = bench._dist_setup(args)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"  # no CUDA here
    bench._barrier(w)
    got = bench._max_over_ranks(10.0 + 5 * rank, w, torch.device("cpu"))
    q.put((rank, got))
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 33500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 15.0), (1, 15.0)]
