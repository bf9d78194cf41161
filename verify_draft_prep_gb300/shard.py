"""Data-parallel sharding of a verify batch by request.

Every step of the path is independent per request (speculative-sampling acceptance, the residual
race and the bonus token read only that request's rows; the draft-batch rebuild reads only that
request's accepted count), so a batch splits over ranks with no exchange on the data path. The
one thing a rank must know about the others is where its requests sit in the global batch: the
Philox counters carry the global request index (``request_base`` of ``sd_verify``), so a batch
verified in shards draws exactly the numbers one device would draw for the whole batch.

The only collective here is a one-off all-gather of the shard sizes when the shard sizes are not
known in advance (ragged shards); it runs on the host process group, outside the step.
"""

from __future__ import annotations


def shard_bounds(batch: int, world: int, rank: int) -> tuple[int, int]:
    """(start, count) of rank's contiguous share of `batch` requests: the first batch % world
    ranks take one request more than the others."""
    if world < 1 or not 0 <= rank < world or batch < 0:
        raise ValueError(f"bad shard: batch={batch} world={world} rank={rank}")
    q, rem = divmod(batch, world)
    start = rank * q + min(rank, rem)
    return start, q + (1 if rank < rem else 0)


def request_base(count: int, group=None) -> tuple[int, int]:
    """(request_base, global batch) for this rank when each rank holds `count` requests of its
    own: all-gathers the counts and returns the exclusive prefix sum at this rank's position.
    Without an initialised process group it is (0, count)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return 0, count
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    mine = torch.tensor([count], dtype=torch.int64)
    if dist.get_backend(group) == "nccl":
        mine = mine.cuda()
    got = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(got, mine, group=group)
    counts = [int(t.item()) for t in got]
    base = sum(counts[:rank])
    total = sum(counts)
    if total > 2**32:
        raise ValueError(f"global batch {total} exceeds the 32-bit Philox request index")
    return base, total


def whole_job_rate(units_per_rank: int, world: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank processed units_per_rank units, and the
    job took as long as its slowest rank (max_ms milliseconds)."""
    if max_ms <= 0:
        raise ValueError("the timed region must have a positive duration")
    return world * units_per_rank / (max_ms / 1e3)
