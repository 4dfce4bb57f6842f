"""Row sharding across ranks (one process per GPU).

Rows are independent units of the selection, so a multi-GPU run splits the
N rows into contiguous, balanced blocks, one per rank, and every rank writes
its own CBSR block. There is no exchange step on the data path: no collective
is needed (weak scaling when each rank keeps a fixed number of rows).
"""
from __future__ import annotations


def row_range(N: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the rows owned by `rank`; blocks differ in size by at most one row."""
    if world < 1 or not (0 <= rank < world) or N < 0:
        raise ValueError("need N >= 0, world >= 1 and 0 <= rank < world")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)
