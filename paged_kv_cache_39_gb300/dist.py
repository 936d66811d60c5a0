"""Process-group plumbing for running the hot path as per-GPU replicas.

The hot path has no exchange step: requests are independent, every GPU owns
its own pool, tables and caches, so N GPUs run N replicas that share nothing
on the data path.  The process group only provides the barrier around the
timed region and the max-over-ranks reduction of the measured time.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass
class Rank:
    rank: int = 0
    local_rank: int = 0
    world_size: int = 1

    @property
    def is_main(self) -> bool:
        return self.rank == 0


def from_env() -> Rank:
    return Rank(int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
                int(os.environ.get("WORLD_SIZE", 1)))


def init(backend: str) -> Rank:
    r = from_env()
    if r.world_size > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29517")
        dist.init_process_group(backend=backend, rank=r.rank, world_size=r.world_size)
    return r


def barrier(device=None) -> None:
    if dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.device(device).index or 0])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard(n: int, r: Rank):
    """Contiguous share [lo, hi) of n independent units for this rank."""
    base, extra = divmod(n, r.world_size)
    lo = r.rank * base + min(r.rank, extra)
    return lo, lo + base + (1 if r.rank < extra else 0)


def finalize() -> None:
    if dist.is_initialized():
        dist.destroy_process_group()
