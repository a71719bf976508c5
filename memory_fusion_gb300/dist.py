"""Multi-rank plumbing of the benchmark: one process per GPU, each running its
own batch of independent rows (weak scaling).  Rows of the fused GEMM +
row-reduce problem are independent, so no collective touches the data path;
the only collectives are the timing barrier and the max over ranks of the
elapsed time.  Works with the nccl backend on GPUs and gloo on CPUs."""
from __future__ import annotations

import os


def env():
    """(world_size, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


class Ranks:
    def __init__(self, backend: str | None = None, device=None):
        self.world, self.rank, self.local = env()
        self.device = device
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            kw = {"device_id": device} if backend == "nccl" and device is not None else {}
            dist.init_process_group(backend or "nccl", **kw)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, value: float) -> float:
        """Max of a float over ranks (the slowest rank sets the job time)."""
        if self.pg is None:
            return float(value)
        import torch
        dev = self.device if self.device is not None else "cpu"
        t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.barrier()
            self.pg.destroy_process_group()
            self.pg = None


def seed_for(base_seed: int, rank: int) -> int:
    """Each rank's batch is its own seeded draw of the workload (rank 0 = base)."""
    return base_seed + 1000 * rank


def job_throughput(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world / seconds_max
