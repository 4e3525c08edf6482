"""Request sharding over replicas: one process per GPU, no collective on the
data path.

The rows of a verify window belong to N requests that share only the weights
(Decode-Verify-Rollback, tgstat @ashnskt post 392, paragraph 4: W = N x K rows
in one fixed-size verify batch), and every row's result is independent of the
rest of the window.  A multi-GPU run therefore replicates the weights and
gives each rank its own block of requests; each rank runs the whole verify
step on its block.  The host gathers the emitted tokens, accept lengths and
rollback points in rank order, and a timing takes the slowest rank.
"""
from __future__ import annotations

import torch


def rank_requests(n_per_rank: int, rank: int) -> range:
    """Global indices of the requests rank ``rank`` owns (weak scaling: every
    rank owns the same number, rank r the block [r * n, (r + 1) * n))."""
    if n_per_rank < 0 or rank < 0:
        raise ValueError("n_per_rank and rank must be >= 0")
    return range(rank * n_per_rank, (rank + 1) * n_per_rank)


def request_ids(indices) -> torch.Tensor:
    """Stable request ids (the Gumbel noise is keyed by them, never by the
    batch slot or the rank that happens to verify the request)."""
    g = torch.as_tensor(list(indices), dtype=torch.int64)
    return (g * 1000 + 17).to(torch.int32)


def gather_in_rank_order(t: torch.Tensor, group=None) -> torch.Tensor:
    """Concatenate one equally shaped tensor per rank, rank 0 first."""
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return t.clone()
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.cat(parts, dim=0)


def slowest(ms: float, device=None, group=None) -> float:
    """The largest of the ranks' times (the job is as fast as its slowest rank)."""
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
