"""Host-side partition of independent KDA problems across ranks (one process per GPU).

Every (sequence, head) problem of the forward pass is independent, so a multi-GPU run splits
whole sequences across ranks and needs no collective on the data path: each rank calls the
library on its own slice, and the results are already where the caller needs them.
"""
from __future__ import annotations


def batch_range(B: int, rank: int, world: int) -> range:
    """Contiguous, balanced split of B sequences (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def packed_ranges(cu_seqlens, world: int) -> list[range]:
    """Splits the sequences of a packed batch into `world` contiguous groups with balanced
    token counts (greedy on the prefix sums). Returns one range of sequence indices per rank."""
    cu = [int(x) for x in cu_seqlens]
    n = len(cu) - 1
    total = cu[-1] - cu[0] if n > 0 else 0
    bounds = [0]
    for r in range(1, world):
        target = cu[0] + total * r / world
        # first sequence boundary at or after the target, never moving backwards
        s = bounds[-1]
        while s < n and cu[s] < target:
            s += 1
        bounds.append(s)
    bounds.append(n)
    return [range(bounds[i], bounds[i + 1]) for i in range(world)]


def local_cu_seqlens(cu_seqlens, seqs: range):
    """Offsets of a contiguous group of packed sequences, rebased to start at 0, and the token
    range [t0, t1) that the group occupies in the packed axis."""
    cu = [int(x) for x in cu_seqlens]
    if len(seqs) == 0:
        return [0], (0, 0)
    t0, t1 = cu[seqs.start], cu[seqs.stop]
    return [c - t0 for c in cu[seqs.start:seqs.stop + 1]], (t0, t1)
