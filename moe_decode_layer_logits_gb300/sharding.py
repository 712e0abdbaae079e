"""Host-side helpers for running the tail on several GPUs as independent
replicas: token rows are independent, so a batch splits by rows with no
exchange on the data path; the only collective is the timing reduction."""

from __future__ import annotations


def token_shard(T: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, stop) rows of a T-row batch for `rank` of `world`;
    the first T % world ranks get one extra row."""
    if world < 1 or not (0 <= rank < world) or T < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float) -> float:
    """Largest `value` over the ranks of the default process group (the
    slowest rank sets a step's time); identity without a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
