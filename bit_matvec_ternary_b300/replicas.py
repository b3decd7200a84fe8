"""Multi-GPU bookkeeping for independent replicas.

The ternary linears have no exchange step between GPUs: a replica on every
rank runs the whole stack on its own batch, and whole-job throughput is the
sum of the ranks' work over the slowest rank's time.  This module holds that
arithmetic and the row split a sharded deployment would use; both run on any
torch.distributed backend (the tests use gloo on CPU).
"""
from __future__ import annotations


def aggregate_throughput(local_ms: float, local_units: float, group=None):
    """(max ms over ranks, sum of units over ranks, units/s) via all_reduce."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return local_ms, local_units, local_units / (local_ms / 1e3)
    t = torch.tensor([local_ms], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    ms, units = float(t.item()), float(u.item())
    return ms, units, units / (ms / 1e3)


def row_shard(M: int, rank: int, world: int, align: int = 16) -> tuple[int, int]:
    """Contiguous output-row range [m0, m1) of `rank`, cut on 16-row panel
    boundaries (a TL2P panel is never split between ranks)."""
    panels = (M + align - 1) // align
    p0 = panels * rank // world
    p1 = panels * (rank + 1) // world
    return min(M, p0 * align), min(M, p1 * align)
