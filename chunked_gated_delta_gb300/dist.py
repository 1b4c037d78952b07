"""Host-side logic for running the KDA forward on several GPUs of one node.

The forward decomposes into independent (sequence, head) units: no unit reads
another's state, so GPUs share work without any collective on the data path.
Two ways to use N GPUs:

* replicas (weak scaling, what ``bench.py --gpus N`` measures): every rank
  runs its own batch of the workload; the job's throughput is the tokens of
  all ranks over the slowest rank's time;
* sharding one batch (strong scaling): :func:`plan_shard` gives each rank a
  contiguous block of sequences (or, with fewer sequences than ranks, of
  heads), :func:`take_shard` cuts the rank's block out of the batch as a
  problem of its own (a batch slice for fixed length; for a packed batch the
  rows of its sequences with ``cu_seqlens`` rebased to start at 0, and the
  matching rows of ``h0``), :func:`fwd_shard` runs the forward on it, and
  :func:`place_shard` writes the block's o and ht into the full tensors.
  Each rank's o and ht are disjoint slices of the whole, so nothing is
  exchanged on the data path.

* one sequence split along T (context parallel), the one layout that needs
  an exchange: :func:`plan_time_shard` gives each rank a contiguous token
  range (on 64-token chunk boundaries); each rank computes its range's affine
  state map [P | Q] (``kda_fwd_state_map``), the maps are all-gathered in rank
  order (K x (K + V) fp32 per sequence and head), ``kda_chain_states``
  composes them into every range's entry state, and each rank finishes its
  range with the scan from its entry state (:func:`fwd_context_parallel`, or
  :func:`context_parallel_maps` / :func:`context_parallel_finish` around an
  exchange of the caller's own).

Only the timing needs communication otherwise: a barrier around the timed
region and a max over ranks of the elapsed time (:func:`max_over_ranks`),
which works on both the gloo (CPU) and NCCL backends.
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


class Shard:
    """One rank's block of a batch: sequences [s0, s1) and heads [h0, h1), with
    the packed token rows [r0, r1) of those sequences (packed batches) or the
    batch rows [s0, s1) (fixed length)."""

    __slots__ = ("s0", "s1", "h0", "h1", "r0", "r1", "varlen")

    def __init__(self, s0, s1, h0, h1, r0, r1, varlen):
        self.s0, self.s1, self.h0, self.h1, self.r0, self.r1, self.varlen = s0, s1, h0, h1, r0, r1, varlen

    def __repr__(self):
        return (f"Shard(seqs=[{self.s0},{self.s1}), heads=[{self.h0},{self.h1}), rows=[{self.r0},{self.r1}), "
                f"varlen={self.varlen})")


def plan_shard(B: int, T: int, H: int, rank: int, world: int, cu_seqlens=None) -> Shard:
    """This rank's block.  Sequences are split into contiguous blocks (each
    rank's inputs and outputs are then contiguous slices); with fewer
    sequences than ranks the heads are split instead.  ``cu_seqlens`` is the
    packed batch's offsets as host integers (a list, or a CPU tensor), or
    None for B fixed-length sequences of T tokens."""
    varlen = cu_seqlens is not None
    cu = [int(c) for c in cu_seqlens] if varlen else None
    N = len(cu) - 1 if varlen else B
    if N >= world:
        s0, s1 = shard_range(N, rank, world)
        hb, he = 0, H
    else:
        s0, s1 = 0, N
        hb, he = shard_range(H, rank, world)
    r0, r1 = (cu[s0], cu[s1]) if varlen else (s0, s1)
    return Shard(s0, s1, hb, he, r0, r1, varlen)


def take_shard(sh: Shard, q, k, v, g, beta, h0=None, cu_seqlens=None):
    """The block's inputs as a problem of its own: (q, k, v, g, beta, h0,
    cu_seqlens).  A block of whole sequences is a slice (no copy, except the
    rebased cu_seqlens); a block of heads is a strided slice and is copied
    into contiguous tensors."""
    if sh.varlen:
        rows = slice(sh.r0, sh.r1)
        q, k, v, g, beta = (t[:, rows] for t in (q, k, v, g, beta))
        cu = cu_seqlens[sh.s0:sh.s1 + 1] - cu_seqlens[sh.s0]
    else:
        b = slice(sh.s0, sh.s1)
        q, k, v, g, beta = (t[b] for t in (q, k, v, g, beta))
        cu = None
    if h0 is not None:
        h0 = h0[sh.s0:sh.s1]
    if (sh.h0, sh.h1) != (0, v.shape[2]):
        hs = slice(sh.h0, sh.h1)
        q, k, v, g = (t[:, :, hs].contiguous() for t in (q, k, v, g))
        beta = beta[:, :, hs].contiguous()
        if h0 is not None:
            h0 = h0[:, hs].contiguous()
    return q, k, v, g, beta, h0, cu


def fwd_shard(sh: Shard, q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, output_final_state=True,
              stream=None):
    """The forward (the library's kda_fwd through the binding) on this rank's
    block; returns the block's (o, ht)."""
    from . import binding
    lq, lk, lv, lg, lb, lh0, lcu = take_shard(sh, q, k, v, g, beta, h0, cu_seqlens)
    return binding.fwd(lq, lk, lv, lg, lb, scale, h0=lh0, cu_seqlens=lcu, output_final_state=output_final_state,
                       stream=stream)


def place_shard(sh: Shard, o_local, ht_local, o, ht=None):
    """Writes a block's (o, ht) into the full outputs (any device; a copy)."""
    rows = slice(sh.r0, sh.r1)
    hs = slice(sh.h0, sh.h1)
    if sh.varlen:
        o[:, rows, hs] = o_local
    else:
        o[rows, :, hs] = o_local
    if ht is not None and ht_local is not None:
        ht[sh.s0:sh.s1, hs] = ht_local


# ---------------------------------------------------------------- context parallel

CHUNK = 64


def plan_time_shard(T: int, rank: int, world: int):
    """This rank's token range [t0, t1) of sequences of T tokens split along T
    across `world` ranks: contiguous, in rank order, on 64-token chunk
    boundaries (every rank's chunks are then chunks of the whole sequence),
    the chunk counts differing by at most one."""
    nt = (T + CHUNK - 1) // CHUNK
    c0, c1 = shard_range(nt, rank, world)
    return min(T, c0 * CHUNK), min(T, c1 * CHUNK)


def context_parallel_maps(q, k, v, g, beta, cu_seqlens=None, stream=None):
    """Pass 1 on this rank's tokens: the affine map [P | Q] of its range for
    every (sequence, head), fp32 [N, H, K, K + V].  Returns (pq, workspace,
    dims); keep the workspace for :func:`context_parallel_finish`."""
    from . import binding
    return binding.state_map(q, k, v, g, beta, cu_seqlens=cu_seqlens, stream=stream)


def context_parallel_finish(pq_all, rank: int, workspace, dims, scale, h0=None, output_final_state=True,
                            stream=None):
    """After the exchange: pq_all [R, N, H, K, K + V] holds every range's map in
    rank order.  Chains them into the entry states, then runs this rank's scan
    from its entry state on the workspace of pass 1.  Returns (o, ht): this
    rank's outputs [B, T_r, H, V] and the state after its range (on the last
    rank, the sequences' final state)."""
    import torch
    from . import binding
    h_in = binding.chain_states(pq_all, h0, stream=stream)
    R, N, H, K, KV = pq_all.shape
    V = KV - K
    o = torch.empty((dims.B, dims.T, H, V), dtype=torch.bfloat16, device=pq_all.device)
    ht = torch.empty((N, H, K, V), dtype=torch.float32, device=pq_all.device) if output_final_state else None
    binding.fwd_scan(scale, h_in[rank], o, ht, dims, workspace, stream)
    return o, ht


def fwd_context_parallel(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, group=None, stream=None):
    """The forward of sequences split along T across the ranks of `group`
    (torch.distributed, one GPU per rank): q, k, v, g, beta (and cu_seqlens)
    hold this rank's tokens of every sequence, the ranks' ranges in rank
    order; h0 is the sequences' initial state (every rank passes the same).
    One all-gather of the maps is the only exchange.  Returns this rank's
    (o, ht) as :func:`context_parallel_finish`."""
    import torch
    import torch.distributed as tdist
    rank, world = tdist.get_rank(group), tdist.get_world_size(group)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    pq, ws, dims = context_parallel_maps(q, k, v, g, beta, cu_seqlens, stream)
    parts = [torch.empty_like(pq) for _ in range(world)]
    tdist.all_gather(parts, pq, group=group)
    return context_parallel_finish(torch.stack(parts), rank, ws, dims, scale, h0, stream=stream)
