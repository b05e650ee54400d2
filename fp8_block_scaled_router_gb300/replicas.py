"""Host logic of multi-GPU runs: independent replicas, one per rank.

The routed MoE layer is data-parallel over tokens and the deployment the pages describe
("NetraRuntime/netra-kernel" README, deployment table: DP8 serving) runs one replica per
GPU with no collective on the layer's data path. Each rank therefore steps through its own
window of the seeded token stream; the only cross-rank traffic is the timing handshake
(barrier, then the slowest rank's elapsed time), which works on any torch.distributed
backend (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations


def token_offset(rank: int, world: int, ntok: int) -> int:
    """First token of rank's window: the stream is cut into `world` equal windows."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    return rank * (ntok // world)


def slowest(elapsed_s: float, dist=None, device=None) -> float:
    """The largest elapsed time over all ranks (the job is as fast as its slowest rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(elapsed_s)
    import torch
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, steps: int, tokens_per_step: int, elapsed_s: float) -> float:
    """Whole-job tokens/s: every rank processed steps * tokens_per_step tokens."""
    if elapsed_s <= 0:
        raise ValueError("elapsed time must be positive")
    return world * steps * tokens_per_step / elapsed_s
