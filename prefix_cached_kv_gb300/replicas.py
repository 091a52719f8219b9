"""Replica plumbing for multi-GPU runs of the library (one process per GPU, launched by torchrun).

The hot path has no exchange step: every rank runs its own queries on its own GPU. A multi-GPU
run therefore only needs a barrier around the timed region, the maximum of the ranks' times and
the whole-job throughput (the units all ranks processed over that maximum). The process group
uses NCCL when the process sees a GPU and gloo otherwise (which is how the CPU tests run it).
"""
from __future__ import annotations

import os

_PG = None   # backend name once the process group is up


def world() -> int:
    """Number of ranks (WORLD_SIZE, 1 when not launched by torchrun)."""
    return int(os.environ.get("WORLD_SIZE", "1"))


def rank() -> int:
    """This process's rank (RANK, 0 when not launched by torchrun)."""
    return int(os.environ.get("RANK", "0"))


def init(backend: str | None = None) -> str | None:
    """Join the process group when there is more than one rank; returns the backend (or None)."""
    global _PG
    if world() <= 1 or _PG is not None:
        return _PG
    import torch
    import torch.distributed as dist
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dist.init_process_group(backend)
    _PG = backend
    return _PG


def barrier() -> None:
    if _PG is not None:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float) -> float:
    """The largest x over all ranks (x itself on one rank)."""
    if _PG is None:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if _PG == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_max: float, n_ranks: int | None = None) -> float:
    """Whole-job rate: every rank processed units_per_rank in at most ms_max milliseconds
    (weak scaling), so the job processed n_ranks * units_per_rank in ms_max."""
    n = world() if n_ranks is None else n_ranks
    return n * units_per_rank / (ms_max * 1e-3)


def finish() -> None:
    global _PG
    if _PG is not None:
        import torch.distributed as dist
        dist.destroy_process_group()
        _PG = None
