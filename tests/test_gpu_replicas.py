"""The replica path with the product's own verify step: two gloo ranks, each
a separate process running libbiv's kernels on the same GPU for its own
block of requests (RMSNorm -> LM head with the fused Gumbel-max selection
and the coupled accept, the tiny workload).  The ranks' kernels never wait
on one another; only the host gathers.  The gathered tokens, accept lengths
and rollback points equal the whole window verified at once by one process,
and the oracle's."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from invariant_verify_gb300 import replicas, synth

pytestmark = pytest.mark.gpu
SEED = synth.PHILOX_SEED
WORLD = 2


def _problem():
    cfg = synth.TINY
    n_total = WORLD * cfg.N
    g = synth.generator(88)
    h = synth.bf16_normal((n_total * cfg.K, cfg.d), cfg.h_std, g)
    lm = synth.bf16_normal((cfg.vocab, cfg.d), cfg.w_std, g)
    p0 = torch.randint(16, 4000, (n_total,), generator=g, dtype=torch.int64).to(torch.int32)
    drafts = torch.randint(0, cfg.vocab, (n_total * cfg.K,), generator=g, dtype=torch.int64).to(torch.int32)
    return cfg, h, lm, p0, drafts


def _gpu_verify(cfg, h, lm, p0, req, drafts):
    """libbiv's verify step of a block of requests (rows request-major)."""
    from invariant_verify_gb300 import abi as B
    n, K = p0.shape[0], cfg.K
    dev = lambda t: t.cuda().contiguous()
    hd, lmd = dev(h), dev(lm)
    hn = torch.empty_like(hd)
    B.biv_rmsnorm(hd, dev(torch.ones(cfg.d, dtype=torch.bfloat16)), hn, cfg.eps)
    pos = (p0.to(torch.int64)[:, None] + torch.arange(K)[None, :]).reshape(-1).to(torch.int32)
    rq = req.repeat_interleave(K).to(torch.int32)
    W = n * K
    tok = torch.empty(W, dtype=torch.int32, device="cuda")
    L = torch.empty(n, dtype=torch.int32, device="cuda")
    nl = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.biv_lm_head_gumbel_workspace_size(W, cfg.vocab, cfg.d), dtype=torch.uint8, device="cuda")
    B.biv_lm_head_gumbel_accept(hn, lmd, dev(rq), dev(pos), SEED, cfg.temperature, tok, dev(drafts), dev(p0), n, K,
                                L, nl, ws)
    torch.cuda.synchronize()
    assert B.biv_device_error() == 0
    return tok.cpu(), L.cpu(), nl.cpu(), hn.cpu()


def _rank_main(rank, port, out_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        torch.cuda.set_device(0)
        cfg, h, lm, p0, drafts = _problem()
        mine = replicas.rank_requests(cfg.N, rank)
        rows = slice(mine.start * cfg.K, mine.stop * cfg.K)
        tok, L, nl, _ = _gpu_verify(cfg, h[rows], lm, p0[mine.start:mine.stop], replicas.request_ids(mine),
                                    drafts[rows])
        got = {"tok": replicas.gather_in_rank_order(tok), "L": replicas.gather_in_rank_order(L),
               "nl": replicas.gather_in_rank_order(nl)}
        if rank == 0:
            torch.save(got, out_path)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_of_the_product_step_match_whole_window(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_verify_gb300 import build
    build.build()
    out = str(tmp_path / "gathered.pt")
    mp.start_processes(_rank_main, args=(_free_port(), out), nprocs=WORLD, join=True, start_method="spawn")
    got = torch.load(out)
    cfg, h, lm, p0, drafts = _problem()
    every = range(WORLD * cfg.N)
    tok, L, nl, hn = _gpu_verify(cfg, h, lm, p0, replicas.request_ids(every), drafts)
    assert torch.equal(got["tok"], tok) and torch.equal(got["L"], L) and torch.equal(got["nl"], nl)
    # and the oracle's selection and accept on the GPU's own fp32 logits
    from invariant_verify_gb300 import abi as B
    logits = torch.empty(hn.shape[0], cfg.vocab, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(hn.cuda(), lm.cuda(), logits)
    pos = (p0.numpy().astype(np.int64)[:, None] + np.arange(cfg.K)[None, :]).reshape(-1).astype(np.int32)
    rq = replicas.request_ids(every).repeat_interleave(cfg.K).numpy()
    ref = oracle.gumbel_argmax(logits.cpu(), rq, pos, SEED, cfg.temperature)
    assert np.array_equal(tok.numpy(), ref)
    rL, rnl = oracle.verify_accept(ref, drafts.numpy(), p0.numpy(), WORLD * cfg.N, cfg.K)
    assert np.array_equal(L.numpy(), rL) and np.array_equal(nl.numpy(), rnl)
