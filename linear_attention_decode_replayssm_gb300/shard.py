"""Which batch rows a rank owns when the decode step runs on several GPUs.

Rows (and heads) of the decode step are independent and the step has no
exchange ("[Kernel] ReplaySSM: cache SSM inputs for faster Gated DeltaNet
standard decode", §Tests: TP2 runs with per-rank sharded caches), so ranks
split the batch into contiguous row blocks, each with its own state pool,
and no collective touches the data path.
"""


def rows_of_rank(global_batch, rank, world):
    """Half-open range [lo, hi) of global rows owned by ``rank``; blocks
    differ in size by at most one row."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError("bad rank/world/global_batch")
    base, extra = divmod(global_batch, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi
