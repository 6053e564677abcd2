"""How the attention path is split across ranks (one process per GPU).

Every (batch, head) pair is an independent problem, so the B*H axis is cut
into contiguous slices, one per rank; each rank reads its slice of Q, K, V
and writes its slice of O and LSE.  No collective touches the data path.
The benchmark instead runs one full-size replica per rank (weak scaling),
each from its own seed.
"""
from __future__ import annotations


def head_slice(num_heads: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the flattened B*H axis owned by `rank`.

    Slices are contiguous, cover every head exactly once, and differ in
    length by at most one.
    """
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if num_heads < 0:
        raise ValueError("num_heads must be >= 0")
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def replica_seed(seed: int, rank: int) -> int:
    """Seed of the independent replica that `rank` runs in the benchmark."""
    return seed + 1000 * rank
