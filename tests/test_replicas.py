"""Multi-replica host path on CPU: two gloo ranks each verify their own block
of requests and the gathered result equals the whole window verified at once
(rows are independent, the noise is keyed by request id, not by rank).  The
per-rank verify step is the oracle's (tiny config: RMSNorm -> LM head ->
Gumbel-max -> accept); the sharding, the gather in rank order and the
slowest-rank timing are the package's own host code."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from invariant_verify_gb300 import replicas, synth

SEED = synth.PHILOX_SEED
WORLD = 2


def _global_problem():
    cfg = synth.TINY
    n_total = WORLD * cfg.N
    g = synth.generator(77)
    h = synth.bf16_normal((n_total * cfg.K, cfg.d), cfg.h_std, g)
    lm = synth.bf16_normal((cfg.vocab, cfg.d), cfg.w_std, g)
    p0 = torch.randint(16, 4000, (n_total,), generator=g, dtype=torch.int64).to(torch.int32)
    mask, ids = synth.draft_errors((n_total, cfg.K), cfg.draft_err, cfg.vocab, seed=78)
    return cfg, h, lm, p0, mask, ids


def _verify(cfg, h, lm, p0, req, mask, ids):
    """Oracle verify step of a block of requests (rows request-major)."""
    n = p0.shape[0]
    K = cfg.K
    y = oracle.round_bf16(oracle.rmsnorm(h, np.ones(cfg.d), cfg.eps))
    logits = oracle.gemm(y, lm).astype(np.float32)
    pos = (p0.numpy().astype(np.int64)[:, None] + np.arange(K)[None, :]).reshape(-1).astype(np.int32)
    tgt = oracle.gumbel_argmax(logits, req.repeat_interleave(K).numpy(), pos, SEED, cfg.temperature)
    draft = synth.apply_draft_errors(torch.from_numpy(tgt), mask.reshape(-1), ids.reshape(-1)).numpy()
    L, new_len = oracle.verify_accept(tgt, draft, p0.numpy(), n, K)
    return tgt.astype(np.int32), L.astype(np.int32), new_len.astype(np.int32)


def _rank_main(rank, port, out_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cfg, h, lm, p0, mask, ids = _global_problem()
        mine = replicas.rank_requests(cfg.N, rank)
        rows = slice(mine.start * cfg.K, mine.stop * cfg.K)
        tgt, L, new_len = _verify(cfg, h[rows], lm, p0[mine.start:mine.stop], replicas.request_ids(mine),
                                  mask[mine.start:mine.stop], ids[mine.start:mine.stop])
        all_tgt = replicas.gather_in_rank_order(torch.from_numpy(tgt))
        all_L = replicas.gather_in_rank_order(torch.from_numpy(L))
        all_nl = replicas.gather_in_rank_order(torch.from_numpy(new_len))
        t = replicas.slowest(10.0 + rank)
        if rank == 0:
            torch.save({"tgt": all_tgt, "L": all_L, "new_len": all_nl, "slowest": t}, out_path)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_rank_requests_partition():
    n = 8
    owned = [i for r in range(4) for i in replicas.rank_requests(n, r)]
    assert owned == list(range(4 * n))
    with pytest.raises(ValueError):
        replicas.rank_requests(-1, 0)


def test_request_ids_do_not_depend_on_rank():
    assert torch.equal(replicas.request_ids(range(3, 5)), replicas.request_ids([3, 4]))
    assert len(set(replicas.request_ids(range(64)).tolist())) == 64


def test_two_gloo_ranks_match_whole_window(tmp_path):
    out = str(tmp_path / "gathered.pt")
    mp.start_processes(_rank_main, args=(_free_port(), out), nprocs=WORLD, join=True, start_method="spawn")
    got = torch.load(out)
    cfg, h, lm, p0, mask, ids = _global_problem()
    every = range(WORLD * cfg.N)
    tgt, L, new_len = _verify(cfg, h, lm, p0, replicas.request_ids(every), mask, ids)
    assert np.array_equal(got["tgt"].numpy(), tgt)
    assert np.array_equal(got["L"].numpy(), L)
    assert np.array_equal(got["new_len"].numpy(), new_len)
    assert got["slowest"] == 11.0
    # the windows differ per rank, so the check is not vacuous
    assert not np.array_equal(tgt[:cfg.N * cfg.K], tgt[cfg.N * cfg.K:])


def _plan_rank_main(rank, port, out_path):
    """One rank of the benchmark's host set-up: its own window plan (the
    request block, ids, contexts, drafter errors), gathered in rank order."""
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cfg = synth.SWEEP
        plan = replicas.rank_window_plan(cfg, 64, 16, rank)
        ids = replicas.gather_in_rank_order(plan["req_ids"])
        ctx = replicas.gather_in_rank_order(plan["ctx"])
        mask = replicas.gather_in_rank_order(plan["draft_mask"].to(torch.int32))
        if rank == 0:
            torch.save({"ids": ids, "ctx": ctx, "mask": mask}, out_path)
    finally:
        dist.destroy_process_group()


def test_bench_rank_windows_disjoint_and_stable(tmp_path):
    """The benchmark's per-rank windows (weak scaling): two gloo ranks build
    their plans; the request ids are disjoint across ranks and are rank r's
    block of the job, and every rank's plan is the same as one built in
    another process (seeded by the rank only)."""
    out = str(tmp_path / "plans.pt")
    mp.start_processes(_plan_rank_main, args=(_free_port(), out), nprocs=WORLD, join=True, start_method="spawn")
    got = torch.load(out)
    cfg = synth.SWEEP
    plans = [replicas.rank_window_plan(cfg, 64, 16, r) for r in range(WORLD)]
    assert torch.equal(got["ids"], torch.cat([p["req_ids"] for p in plans]))
    assert torch.equal(got["ctx"], torch.cat([p["ctx"] for p in plans]))
    assert torch.equal(got["mask"], torch.cat([p["draft_mask"].to(torch.int32) for p in plans]))
    ids = got["ids"].tolist()
    assert len(set(ids)) == len(ids) == WORLD * 64
    assert torch.equal(got["ids"][64:], replicas.request_ids(range(64, 128)))
    # the ranks' contexts follow the workload recipe and differ between ranks
    c = got["ctx"]
    assert int(c.min()) >= cfg.ctx_lo and int(c.max()) <= cfg.ctx_hi
    assert not torch.equal(c[:64], c[64:])
