"""Multi-GPU partition of the DSA decode step (one process per GPU).

The decode step is independent per request: every request's index-K pages, logits, top-k and
attention touch only that request's data.  The N-GPU configuration therefore shards requests (or
whole batches) across ranks with no collective on the data path; ranks meet only for timing (a
barrier and a max-reduction of the step time).  Per-rank work is fixed as N grows (weak scaling).

Helpers here are host-side bookkeeping only (which requests or which batch a rank owns, the
slowest rank's time); all computation stays in the CUDA library.
"""
from __future__ import annotations

import os
from typing import List, Optional

import torch
import torch.distributed as dist

from . import workloads


def env_rank_world():
    """(rank, world_size, local_rank) from the torchrun environment (defaults: single process)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_requests(num_requests: int, rank: int, world: int) -> List[int]:
    """Requests owned by `rank` when one batch is split across `world` ranks: a contiguous block,
    the first (num_requests % world) ranks taking one extra request."""
    base, extra = divmod(num_requests, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return list(range(lo, hi))


def rank_workload(name: str, rank: int) -> workloads.Workload:
    """The batch a rank runs in the weak-scaling benchmark: the named workload's shape, with its own
    seed (seed + 1000 * rank) so that ranks process different data."""
    wl = workloads.make(name)
    if rank == 0:
        return wl
    return workloads.make_custom(wl.name, wl.seed + 1000 * rank, wl.seq_lens, wl.q_lens, wl.topk, wl.heads,
                                 pool_pages=wl.num_pages)


def max_over_ranks(value: float, device: Optional[torch.device] = None) -> float:
    """Maximum of a per-rank scalar over all ranks (identity without an initialised group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(rows_per_rank: int, world: int, slowest_ms: float) -> float:
    """Whole-job throughput: every rank's query rows over the slowest rank's step time."""
    return rows_per_rank * world / (slowest_ms / 1000.0)
