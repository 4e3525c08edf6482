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


def rank_window_plan(cfg, n_per_rank: int, K: int, rank: int) -> dict:
    """The seeded, host-side description of rank ``rank``'s verify window:
    its requests' global indices and stable ids, cached context lengths, last
    committed tokens and where its drafter errs (with the ids it then
    proposes).  Everything is drawn from seeds that depend on the rank, so the
    ranks' windows differ, and on nothing else, so a rank's window is the same
    in every run and on every host."""
    from . import synth
    mine = rank_requests(n_per_rank, rank)
    seed = cfg.seed + 1009 * rank
    ctx = synth.context_lengths(cfg, n_per_rank, seed=seed + 100)
    g = synth.generator(seed + 300)
    last = torch.randint(0, cfg.vocab, (n_per_rank,), generator=g, dtype=torch.int64).to(torch.int32)
    mask, ids = synth.draft_errors((n_per_rank, K), cfg.draft_err, cfg.vocab, seed=seed + 400)
    return {"requests": mine, "req_ids": request_ids(mine), "ctx": ctx, "last": last,
            "draft_mask": mask, "draft_ids": ids, "kv_seed": seed + 200}
