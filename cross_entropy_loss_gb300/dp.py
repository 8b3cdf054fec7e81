"""Host-side data-parallel helpers for the cross-entropy path.

Rows are independent, so data parallelism shards rows across ranks and needs no
collective on the data path.  The one real exchange is the denominator of a
per-token mean across ranks -- the "--loss_across_gpus mean token" averaging of
the LossAccelerationPlugin (fms-hf-tuning PR #280, "Early Version Of This
Plugin"): every rank divides by the global count of non-ignored tokens, which it
passes to the C ABI as ``denom``.  These helpers are plain torch.distributed
calls; any backend works (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations


def shard_rows(n_rows: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous row range [begin, end) of ``rank``; sizes differ by at most one row."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(n_rows, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def global_denominator(local_n_valid: int, group=None, device=None) -> float:
    """Sum of every rank's valid-token count (the shared ``denom`` of a per-token mean)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([int(local_n_valid)], dtype=torch.int64, device=device)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def global_loss(local_loss: float, group=None, device=None) -> float:
    """Sum of the ranks' partial losses; with a shared ``denom`` this is the global mean."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_loss)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def max_over_ranks(value: float, group=None, device=None) -> float:
    """Largest value over ranks (a step's wall time is the slowest rank's)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
