"""Replica coordination for runs on N GPUs of one node, one process per GPU.

The layer needs no exchange between GPUs (each GPU runs its own copies of the
layers on its own inputs: replicas), so the only cross-process steps are the
ones a measurement needs: a barrier on both sides of a timed region and the
maximum of the ranks' elapsed times. Rank, world size and the rendezvous come
from the environment that torch.distributed.run sets (RANK, WORLD_SIZE,
LOCAL_RANK, MASTER_ADDR, MASTER_PORT). The backend is NCCL for CUDA devices
and gloo on the CPU (the tests run two gloo ranks).
"""

from __future__ import annotations

import os


class Replicas:
    def __init__(self, backend: str | None = None, device=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.device = device
        self._dist = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if device is not None and torch.device(device).type == "cuda" else "gloo"
            kw = {}
            if backend == "nccl":
                kw["device_id"] = torch.device(device)
            if not dist.is_initialized():
                dist.init_process_group(backend, **kw)
            self._dist = dist

    def barrier(self) -> None:
        if self._dist is not None:
            self._dist.barrier()

    def max(self, v: float) -> float:
        """The largest value over the ranks (every rank gets it)."""
        if self._dist is None:
            return float(v)
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64, device=self.device)
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX)
        return float(t.item())

    def throughput(self, units_per_rank: float, elapsed_s: float) -> float:
        """Whole-job rate: the units all ranks processed over the slowest rank's time."""
        return self.world * units_per_rank / self.max(elapsed_s)

    def close(self) -> None:
        if self._dist is not None and self._dist.is_initialized():
            self._dist.destroy_process_group()
