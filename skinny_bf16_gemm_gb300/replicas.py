"""Host-side logic of running the path as independent replicas, one per GPU.

The drafter path has no exchange step on one node here (the TP all-reduce is
represented by local slots), so N GPUs run N independent copies of the same
workload with distinct seeds. A run's time is the slowest rank's, and its
throughput is the work of all ranks over that time (weak scaling).
"""
import os


def rank_info():
    """(rank, world_size, local_rank) from the torchrun environment (1 GPU: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(base_seed: int, rank: int) -> int:
    """Distinct, stable seed per rank."""
    return (int(base_seed) * 1_000_003 + 7919 * int(rank)) & ((1 << 63) - 1)


def slowest_ms(ms: float, device=None) -> float:
    """Max of `ms` over all ranks of the default process group (itself alone if
    no group is initialised). Works with NCCL (device tensor) and gloo (CPU)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(bytes_per_rank_step: int, steps: int, slowest_ms_total: float,
                         world: int) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (slowest_ms_total * 1e-3) / 1e9
