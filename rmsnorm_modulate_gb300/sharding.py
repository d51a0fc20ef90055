"""Row sharding across ranks (one process per GPU).

Every row of every operation here is independent, so a multi-GPU run needs
no data-path collective: each rank normalises a contiguous range of the
B*S rows.  A range that crosses a batch boundary is cut there, so every
segment is one call with a single modulation row (per-batch scale/shift).
"""
from __future__ import annotations


def row_range(rows: int, rank: int, world: int) -> tuple[int, int]:
    """Balanced contiguous range [r0, r1) of `rows` for `rank` of `world`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(rows, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def row_segments(B: int, S: int, rank: int, world: int) -> list[tuple[int, int, int]]:
    """This rank's rows of a [B, S, D] tensor as (batch, s0, s1) segments."""
    r0, r1 = row_range(B * S, rank, world)
    segs = []
    r = r0
    while r < r1:
        b, s = divmod(r, S)
        s1 = min(S, s + (r1 - r))
        segs.append((b, s, s1))
        r += s1 - s
    return segs
