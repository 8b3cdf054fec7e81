"""Host-side data-parallel helpers for the cross-entropy path.

Rows are independent, so data parallelism shards rows across ranks and needs no
collective on the data path.  The one real exchange is the denominator of a
per-token mean across ranks -- the "--loss_across_gpus mean token" averaging of
the LossAccelerationPlugin (fms-hf-tuning PR #280, "Early Version Of This
Plugin"): every rank divides by the global count of non-ignored tokens, which it
passes to the C ABI as ``denom``.  These helpers are plain torch.distributed
calls; any backend works (NCCL on GPUs, gloo on CPU).

``fused_step`` is the step a data-parallel job runs: count the local valid tokens,
sum the counts over ranks in place (on the device with NCCL), run the fused
forward+backward dividing by that total, and sum the ranks' partial losses.
``launch_argv`` / ``relaunch`` start one process per GPU under
``torch.distributed.run``; ``rank_env`` reads the rank layout it sets.
"""
from __future__ import annotations

import os
import socket
import subprocess
import sys


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


def fused_step(count_fn, fused_fn, logits, labels, group=None):
    """One data-parallel step of the per-token mean across ranks.

    ``count_fn(labels)`` returns this rank's valid-token count as a one-element int64
    tensor on the data's device; it is summed over ranks in place before anything
    divides by it, so no gradient is written with a partial denominator.
    ``fused_fn(logits, labels, denom_count)`` runs the fused forward+backward with that
    total as D and returns a dict whose "loss" tensor is this rank's share
    sum(l_i) / D; the shares are summed over ranks, so every rank ends with the
    global mean.  With no process group initialised this is the one-rank step.
    Returns fused_fn's dict plus "denom" (the summed count).
    """
    import torch.distributed as dist

    live = dist.is_available() and dist.is_initialized()
    cnt = count_fn(labels)
    if live:
        dist.all_reduce(cnt, op=dist.ReduceOp.SUM, group=group)
    out = fused_fn(logits, labels, cnt)
    if live:
        dist.all_reduce(out["loss"], op=dist.ReduceOp.SUM, group=group)
    out["denom"] = cnt
    return out


def rank_env() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) as torch.distributed.run exports them (1 process if unset)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank layout: RANK={rank} WORLD_SIZE={world}")
    return rank, world, local


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_argv(nproc: int, script: str, argv: list[str], port: int, python: str | None = None) -> list[str]:
    """Command line that starts ``script argv`` once per local GPU (one node, rendezvous on 127.0.0.1)."""
    if nproc < 1:
        raise ValueError("nproc must be >= 1")
    return [python or sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
            "--master-addr", "127.0.0.1", f"--master-port={port}", script, *argv]


def relaunch(nproc: int, script: str, argv: list[str]) -> int:
    """Run ``script argv`` as ``nproc`` ranks and return the launcher's exit status."""
    return subprocess.call(launch_argv(nproc, script, argv, free_port()))
