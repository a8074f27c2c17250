"""Context parallelism for KDA over T-segments (KCP).

Kimi K3 wiki, "Glossaire", entry "KCP": each rank sends two quantities, the cumulative
transition M and the local state S~ of its stretch of tokens; they compose associatively, the
exchange has a fixed size, and the result is exact ("Notations mathématiques", rows M_t and S~).

Rank r of a group of W ranks holds tokens [r T_r, (r + 1) T_r) of every sequence of the batch
(q, k, v, g, beta shaped [B, T_r, H, d] on its device). One forward pass is:

  1. (M_r, S~_r) of the local segment, for every (sequence, head): the library's transition pass.
  2. One all-gather of the fixed-size pairs (2 x B x H x d_k x d fp32 per rank).
  3. The incoming state of the local segment, S_in(r) = M_{r-1}(... (M_0 S0 + S~_0) ...) + S~_{r-1},
     from the gathered pairs with the library's scan (S0 is the batch's initial state, the same
     on every rank).
  4. The local segment from S_in(r): outputs for the local tokens and, on the last rank, the
     final state of the whole sequence.

The steps are separate functions so that one process can emulate the ranks one after another
(:func:`emulate`: the exchange is then a list), and so that the arithmetic can be swapped for
another implementation (the CPU tests use the oracle's) while the exchange logic stays the same.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import torch


@dataclass
class Ops:
    """The three computations of a KCP pass.

    transitions(k, v, g, beta) -> (M [B, H, dk, dk], S_tilde [B, H, dk, dv])
    scan(Ms [n, B, H, dk, dk], Sts [n, B, H, dk, dv], S0 or None) -> S_in [n + 1, B, H, dk, dv]
    forward(q, k, v, g, beta, S_in) -> (out [B, T_r, H, dv], S_final [B, H, dk, dv])
    """
    transitions: Callable
    scan: Callable
    forward: Callable


def library_ops(C: int = 64, stream=None) -> Ops:
    """The three computations on the GPU through the C ABI (`libkda.so`)."""
    import gated_delta_rule_167_b300 as kda

    def transitions(k, v, g, beta):
        B, T, H, dk = k.shape
        dv = v.shape[-1]
        M = torch.empty(1, B, H, dk, dk, dtype=torch.float32, device=k.device)
        St = torch.empty(1, B, H, dk, dv, dtype=torch.float32, device=k.device)
        kda.kda_segment_transitions(k, v, g, beta, M, St, seg_len=max(T, 1), C=C, stream=stream)
        return M[0], St[0]

    def scan(Ms, Sts, S0):
        n, B, H, dk, dv = Sts.shape
        S_in = torch.empty(n + 1, B, H, dk, dv, dtype=torch.float32, device=Sts.device)
        kda.kda_segment_scan(Ms.contiguous(), Sts.contiguous(), S0, S_in, stream=stream)
        return S_in

    def forward(q, k, v, g, beta, S_in):
        return kda.chunk_fwd(q, k, v, g, beta, S_in, C=C, stream=stream)

    return Ops(transitions, scan, forward)


def local_pair(ops: Ops, k, v, g, beta):
    """Step 1: (M, S~) of this rank's segment, stacked as one [2, ...] exchange buffer when
    d_k = d_v (the supported head sizes)."""
    M, St = ops.transitions(k, v, g, beta)
    return torch.stack([M, St])


def incoming_state(ops: Ops, pairs, rank: int, S0):
    """Step 3: the state entering segment `rank`, from the pairs of the ranks before it
    (pairs[i] is rank i's [2, B, H, d, d] buffer; later entries are not read)."""
    if rank == 0:
        if S0 is not None:
            return S0
        p = pairs[0]
        return torch.zeros(p.shape[1:], dtype=p.dtype, device=p.device)
    Ms = torch.stack([pairs[i][0] for i in range(rank)])
    Sts = torch.stack([pairs[i][1] for i in range(rank)])
    return ops.scan(Ms, Sts, S0)[rank]


def forward(q, k, v, g, beta, S0=None, ops: Optional[Ops] = None, group=None):
    """One KCP forward pass on this rank (steps 1-4 of the module docstring). Every rank of
    `group` calls it with its own segment; returns (out for the local tokens, the state after
    the local segment), which on the last rank is the final state of the sequences."""
    import torch.distributed as dist

    ops = ops or library_ops()
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    mine = local_pair(ops, k, v, g, beta).contiguous()
    pairs = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(pairs, mine, group=group)
    S_in = incoming_state(ops, pairs, rank, S0)
    return ops.forward(q, k, v, g, beta, S_in)


def emulate(q, k, v, g, beta, world: int, S0=None, ops: Optional[Ops] = None):
    """All ranks of a KCP pass in one process: the batch's T axis is cut into `world` equal
    segments (T divisible by `world`), the ranks run steps 1-4 one after another and the
    exchange is a list. Returns (out over all T, final state)."""
    ops = ops or library_ops()
    T = q.shape[1]
    if T % world:
        raise ValueError("T must be divisible by the number of emulated ranks")
    Tr = T // world
    seg = [slice(r * Tr, (r + 1) * Tr) for r in range(world)]

    def part(x, r):
        return x[:, seg[r]].contiguous()

    pairs = [local_pair(ops, part(k, r), part(v, r), part(g, r), part(beta, r))
             for r in range(world)]
    outs, Sf = [], None
    for r in range(world):
        S_in = incoming_state(ops, pairs, r, S0)
        o, Sf = ops.forward(part(q, r), part(k, r), part(v, r), part(g, r), part(beta, r), S_in)
        outs.append(o)
    return torch.cat(outs, dim=1), Sf
