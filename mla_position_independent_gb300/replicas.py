"""Host-side helpers for running the path on several GPUs as independent replicas.

The reconstruction shards by request with no exchange step (every request's chunk table,
row store and queries are independent), so N GPUs run N replicas: each rank takes a
contiguous share of the requests (or its own batch), and the benchmark reduces its timing
with a max over ranks.  No data-path collective exists.
"""
from __future__ import annotations

import numpy as np


def request_shard(B: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) share of B requests for `rank` (sizes differ by at most one)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(B, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def subtable(chunks: np.ndarray, indptr: np.ndarray, lo: int, hi: int):
    """Chunk table of requests [lo, hi) with indptr re-based to start at 0."""
    c0, c1 = int(indptr[lo]), int(indptr[hi])
    sub = np.ascontiguousarray(chunks[c0:c1])
    ip = (np.asarray(indptr[lo:hi + 1], np.int64) - c0).astype(np.int32)
    return sub, ip


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Slowest rank's value (the job's time); identity for a single process."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
