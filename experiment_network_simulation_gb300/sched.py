"""Host-side scheduling of experiment batches: waves that fit an HBM budget,
shards across GPUs, and the gather of per-shard results.

Experiments are independent (the Multiverse page, section 5, "multi-GPU":
each GPU runs its own experiments and cross-GPU execution is independent),
so sharding needs no collective on the simulation path; only the results
are gathered to rank 0 at the end.
"""
from __future__ import annotations

import numpy as np

from . import inputs as I

PER_EXP_KEYS = ("status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
                "msgs_delivered", "digest", "rec_count")


def shard(n: int, rank: int, world: int) -> range:
    """Contiguous slice of n experiments for `rank` of `world` (sizes differ by
    at most one, earlier ranks take the extra)."""
    q, r = divmod(n, world)
    lo = rank * q + min(rank, r)
    return range(lo, lo + q + (1 if rank < r else 0))


def plan_waves(batch: I.Batch, budget_bytes: int, workspace_bytes) -> list:
    """Split the batch, in order, into waves whose workspace fits the budget.
    `workspace_bytes(packed)` sizes a candidate wave (the library's
    mv_workspace_bytes); sizes are monotone in the number of experiments."""
    waves, start, n = [], 0, len(batch)
    while start < n:
        lo, hi = 1, n - start
        if workspace_bytes(batch.subset(range(start, start + 1)).pack()) > budget_bytes:
            raise ValueError(f"experiment {start} alone exceeds the budget")
        while lo < hi:                                  # largest count that fits
            mid = (lo + hi + 1) // 2
            if workspace_bytes(batch.subset(range(start, start + mid)).pack()) <= budget_bytes:
                lo = mid
            else:
                hi = mid - 1
        waves.append(range(start, start + lo))
        start += lo
    return waves


def concat_results(parts: list) -> dict:
    """Join per-experiment and per-node result arrays of consecutive slices."""
    out = {}
    for k in PER_EXP_KEYS:
        out[k] = np.concatenate([p[k] for p in parts])
    for k in ("node_start", "node_end"):
        out[k] = np.concatenate([p[k][: p["node_offset"][-1]] for p in parts])
    off = [0]
    for p in parts:
        off += list(off[-1] + np.asarray(p["node_offset"][1:]))
    out["node_offset"] = np.array(off, np.int64)
    return out


def run_sharded(batch: I.Batch, simulate, rank: int = 0, world: int = 1, group=None) -> dict | None:
    """Simulate this rank's shard with `simulate(packed) -> results` and
    gather every shard's results on rank 0 (None on the other ranks)."""
    mine = shard(len(batch), rank, world)
    res = simulate(batch.subset(mine).pack()) if len(mine) else None
    part = None if res is None else {k: np.asarray(res[k]) for k in PER_EXP_KEYS + (
        "node_start", "node_end", "node_offset")}
    if world == 1:
        return concat_results([part]) if part is not None else None
    import torch.distributed as dist

    parts = [None] * world if rank == 0 else None
    dist.gather_object(part, parts, dst=0, group=group)
    if rank != 0:
        return None
    return concat_results([p for p in parts if p is not None])
