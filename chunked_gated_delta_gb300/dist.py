"""Host-side logic for running the KDA forward on several GPUs of one node.

The forward decomposes into independent (sequence, head) units: no unit reads
another's state, so GPUs share work without any collective on the data path.
Two ways to use N GPUs:

* replicas (weak scaling, what ``bench.py --gpus N`` measures): every rank
  runs its own batch of the workload; the job's throughput is the tokens of
  all ranks over the slowest rank's time;
* sharding one batch (strong scaling): :func:`shard_range` gives each rank a
  contiguous block of sequences (or of heads); each rank writes a disjoint
  slice of o and ht.

Only the timing needs communication: a barrier around the timed region and a
max over ranks of the elapsed time (:func:`max_over_ranks`), which works on
both the gloo (CPU) and NCCL backends.
"""
from __future__ import annotations

import os


def rank_info():
    """(rank, world_size, local_rank) from the torchrun environment (defaults 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_range(n_units: int, rank: int, world: int):
    """Contiguous [start, end) block of n_units for this rank; blocks differ in
    size by at most one and tile [0, n_units) exactly."""
    if world < 1 or not (0 <= rank < world) or n_units < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(x: float, world: int) -> float:
    """Max of a float over all ranks (identity for world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(units_per_rank, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return float(sum(units_per_rank)) / max_seconds
