"""KCP (context parallelism over T-segments) exchange logic, on the CPU.

The orchestration of `gated_delta_rule_167_b300.kcp` (local pair, one fixed-size all-gather,
incoming state from the ranks before, local forward) runs with two gloo ranks, each holding one
half of the sequences' tokens. The arithmetic of the three steps is the oracle's here: the
transition of a segment by definition (the recurrence from S0 = I with v = 0 gives the product
of its M_t; from S0 = 0 it gives S~), the composition rule of (M, S~) pairs, and the recurrence
itself. The stitched result must equal the recurrence over the whole sequence to fp64 rounding.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

NAMES = ("q", "k", "v", "g", "beta")


def oracle_ops():
    import oracle
    from oracle import chunkwise

    from gated_delta_rule_167_b300 import kcp

    def np64(t):
        return None if t is None else t.detach().to(torch.float64).numpy()

    def transitions(k, v, g, beta):
        B, T, H, dk = k.shape
        eye = np.broadcast_to(np.eye(dk), (B, H, dk, dk)).copy()
        kk, vv, gg, bb = map(np64, (k, v, g, beta))
        _, M = oracle.recurrent(kk, kk, np.zeros_like(vv), gg, bb, eye, nthreads=1)
        _, St = oracle.recurrent(kk, kk, vv, gg, bb, None, nthreads=1)
        return torch.from_numpy(M), torch.from_numpy(St)

    def scan(Ms, Sts, S0):
        n, B, H, dk, dv = Sts.shape
        out = np.zeros((n + 1, B, H, dk, dv))
        for b in range(B):
            for h in range(H):
                pair = (np.eye(dk), np.zeros((dk, dv)) if S0 is None else np64(S0[b, h]))
                out[0, b, h] = pair[1]
                for s in range(n):
                    pair = chunkwise.compose((np64(Ms[s, b, h]), np64(Sts[s, b, h])), pair)
                    out[s + 1, b, h] = pair[1]
        return torch.from_numpy(out)

    def forward(q, k, v, g, beta, S_in):
        o, S = oracle.recurrent(*map(np64, (q, k, v, g, beta)), np64(S_in), nthreads=1)
        return torch.from_numpy(o), torch.from_numpy(S)

    return kcp.Ops(transitions, scan, forward)


def _inputs(T=48, seed=4):
    import kda_synth

    return kda_synth.make_prefill_inputs(2, T, 3, 16, 16, "f32", seed=seed, S0_std=0.2)


def _reference(inp):
    import oracle

    return oracle.recurrent(*(inp[n].double().numpy() for n in NAMES),
                            inp["S0"].double().numpy(), nthreads=1)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from gated_delta_rule_167_b300 import kcp

    inp = _inputs()
    T = inp["q"].shape[1]
    Tr = T // world
    mine = {n: inp[n][:, rank * Tr:(rank + 1) * Tr].double().contiguous() for n in NAMES}
    out, S = kcp.forward(*(mine[n] for n in NAMES), S0=inp["S0"].double(), ops=oracle_ops())
    outs = [None] * world
    dist.all_gather_object(outs, (rank, out.numpy(), S.numpy()))
    if rank == 0:
        o_ref, S_ref = _reference(inp)
        got = np.concatenate([o for _, o, _ in sorted(outs, key=lambda x: x[0])], axis=1)
        err_o = float(np.abs(got - o_ref).max())
        err_S = float(np.abs(outs[-1][2] - S_ref).max())
        q.put((err_o, err_S))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_stitch_the_exact_result():
    import oracle

    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 31500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    err_o, err_S = q.get(timeout=5)
    assert err_o < 1e-10 and err_S < 1e-10, (err_o, err_S)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_emulated_ranks_are_exact(world):
    """The single-process emulation (exchange as a list) over 1-4 segments."""
    from gated_delta_rule_167_b300 import kcp

    inp = _inputs(T=48, seed=world)
    x = [inp[n].double() for n in NAMES]
    out, S = kcp.emulate(*x, world=world, S0=inp["S0"].double(), ops=oracle_ops())
    o_ref, S_ref = _reference(inp)
    assert np.abs(out.numpy() - o_ref).max() < 1e-10
    assert np.abs(S.numpy() - S_ref).max() < 1e-10


def test_incoming_state_of_rank_zero_is_S0_or_zero():
    from gated_delta_rule_167_b300 import kcp

    ops = oracle_ops()
    pairs = [torch.zeros(2, 1, 1, 4, 4)]
    S0 = torch.ones(1, 1, 4, 4)
    assert torch.equal(kcp.incoming_state(ops, pairs, 0, S0), S0)
    assert not kcp.incoming_state(ops, pairs, 0, None).any()
