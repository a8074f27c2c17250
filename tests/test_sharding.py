"""Multi-rank partition of independent problems, exercised with 2 gloo ranks on the CPU.

Each rank runs its own share of sequences (here through the CPU oracle, which stands in for a
GPU per rank); the shares are gathered only to check that the union equals a single-process
run. The data path itself has no collective.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_delta_rule_167_b300 import shard


def test_batch_range_covers_everything_once():
    for B in (0, 1, 5, 8, 13):
        for world in (1, 2, 3, 8):
            got = [i for r in range(world) for i in shard.batch_range(B, r, world)]
            assert got == list(range(B))
            sizes = [len(shard.batch_range(B, r, world)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1


def test_packed_ranges_balance_and_cover():
    cu = [0, 11185, 30139, 83195, 90836, 93867, 110864, 118982, 131072]
    for world in (1, 2, 4, 8):
        parts = shard.packed_ranges(cu, world)
        seqs = [s for p in parts for s in p]
        assert seqs == list(range(len(cu) - 1))
        assert all(p.stop == q.start for p, q in zip(parts, parts[1:]))
    local, (t0, t1) = shard.local_cu_seqlens(cu, range(2, 5))
    assert local[0] == 0 and (t0, t1) == (30139, 93867) and local[-1] == t1 - t0


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import kda_synth
    import oracle

    B, T, H, d = 5, 40, 2, 16
    inp = kda_synth.make_prefill_inputs(B, T, H, d, d, "f32", seed=3, S0_std=0.1)
    mine = shard.batch_range(B, rank, world)
    sl = slice(mine.start, mine.stop)
    x = [kda_synth.to_f64_numpy(inp[n][sl]) for n in ("q", "k", "v", "g", "beta")]
    o, S = oracle.recurrent(*x, kda_synth.to_f64_numpy(inp["S0"][sl]), nthreads=1)
    outs = [None] * world
    dist.all_gather_object(outs, (mine.start, o, S))
    if rank == 0:
        full_o, full_S = oracle.recurrent(*(kda_synth.to_f64_numpy(inp[n]) for n in
                                            ("q", "k", "v", "g", "beta")),
                                          kda_synth.to_f64_numpy(inp["S0"]), nthreads=1)
        ok = True
        for start, o_r, S_r in outs:
            n = o_r.shape[0]
            ok &= np.array_equal(o_r, full_o[start:start + n])
            ok &= np.array_equal(S_r, full_S[start:start + n])
        ok &= sum(o_r.shape[0] for _, o_r, _ in outs) == B
        q.put(bool(ok))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_single_process():
    import oracle

    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) is True
