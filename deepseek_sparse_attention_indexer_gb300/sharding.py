"""How the path spreads over several GPUs: replicas on disjoint query rows.

Every query row of the path depends only on its own query and on the shared,
read-only caches: the indexer score row S[i, :] uses query i's indexer heads
and weights with every key, the selection of row i reads only S[i, :], and the
attention of row i reads only q[i] and the latent rows row i selected.  So a
prefill chunk splits into contiguous blocks of query rows, one per GPU, with the
caches replicated and no exchange step; a batch of decode sequences splits by
sequence the same way.  A caller that needs the outputs in one place gathers
them afterwards.  Host logic only: the work on each GPU is the ordinary library
calls on its rows.
"""
from __future__ import annotations


def shard_rows(L: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [start, stop) of L for `rank` of `world`: contiguous blocks, sizes differing by at
    most one, earlier ranks taking the extra rows; empty when L < world for the last ranks."""
    if world < 1 or not 0 <= rank < world or L < 0:
        raise ValueError(f"bad shard request L={L} world={world} rank={rank}")
    base, extra = divmod(L, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_prefill_positions(p0: int, L: int, world: int, rank: int) -> tuple[int, int, int]:
    """(start, stop, q_pos0) of `rank`'s block of a prefill chunk whose first query sits at
    position p0: query row i keeps its position p0 + i, so the block starts at p0 + start."""
    start, stop = shard_rows(L, world, rank)
    return start, stop, p0 + start
