"""Row sharding of the fused epilogues across ranks (host logic only).

Every op is per element or per row, so a [rows, cols] activation splits into
contiguous row blocks with no exchange.  The dropout mask stays the mask of
the unsharded tensor when each shard passes the global flat index of its
first element as `elem_base` (the mask is a function of (seed, offset,
global index) only).
"""


def row_shard(rows: int, world: int, rank: int):
    """Contiguous, balanced split: rank gets rows [start, stop)."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("need rows >= 0 and 0 <= rank < world")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_elem_base(row_start: int, cols: int, global_base: int = 0) -> int:
    """Global flat index of element (row_start, 0) of a [rows, cols] tensor."""
    return global_base + row_start * cols
