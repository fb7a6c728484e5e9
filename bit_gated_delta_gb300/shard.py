"""Data-parallel placement over ranks (one process per GPU).

The decode step, the flush and the prefill are independent per (sequence, head), so the batch is split into
contiguous per-rank slices and no collective runs on the data path. The one exchange the method has is offline:
the head ranking E_h = e_h / (1 - a_h^(2 dP)) ([P1] 무엇과 다른가: the quarter of heads with the largest E_h
stay at 8 bits) must be computed from the calibration error energy of *all* sequences, so every rank sums its
per-head energy before the ranking and all ranks keep the same int8 heads.
"""
from __future__ import annotations

import numpy as np


def batch_slice(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """(first sequence, count) of rank `rank`: contiguous, sizes differ by at most one, lower ranks larger."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError(f"bad placement: batch {global_batch}, world {world}, rank {rank}")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def max_over_ranks(x: float, dist=None) -> float:
    """The largest value of x over all ranks (a step time: the job is as slow as its slowest rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=_device(dist))
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def global_head_energy(e_sum_local, n_local: int, dist=None) -> np.ndarray:
    """Mean per-head calibration error energy over every sequence of every rank.

    e_sum_local: per-head sums of ||Q(S) - S||_F^2 over this rank's n_local sequences."""
    e = np.asarray(e_sum_local, dtype=np.float64)
    n = float(n_local)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        import torch
        t = torch.tensor(np.concatenate([e, [n]]), dtype=torch.float64, device=_device(dist))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        v = t.cpu().numpy()
        e, n = v[:-1], float(v[-1])
    if n <= 0:
        raise ValueError("no calibration sequences")
    return e / n


def assign_heads_global(e_sum_local, n_local: int, a_h, dP: int, frac: float = 0.25, dist=None) -> np.ndarray:
    """Int8-head mask from the energy of all ranks' sequences; identical on every rank."""
    from . import pace_assign_heads
    e = global_head_energy(e_sum_local, n_local, dist)
    return pace_assign_heads(e.astype(np.float32), np.asarray(a_h, dtype=np.float32), dP, frac)


def _device(dist):
    import torch
    return torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
