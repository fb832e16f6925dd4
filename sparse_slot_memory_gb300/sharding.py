"""Host-side split of a workload across GPUs.

The forward shards by stream with no exchange: stream p owns bank rows [p*S, (p+1)*S) and its
chunks c = ti * P + p touch nothing else (phase1_cuda.py, p1_keys_zw_kernel: each chunk's ids are
stream-local). Rank r of G takes a contiguous block of streams and runs Phase 1 + DW on them
alone; the only collectives a multi-GPU run needs are for measurement (a barrier, the max of
the ranks' times).
"""

from __future__ import annotations


def shard_streams(P: int, rank: int, world: int) -> range:
    """Streams of rank `rank` among `world` ranks: contiguous, sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    base, extra = divmod(P, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))
