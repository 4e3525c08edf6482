"""Parity at the workloads' full sizes, in the configuration bench.py and the
verifier use: every selected token and accept length bit-exact against the
oracle, dense outputs on sampled elements the oracle computes one by one,
and rows bitwise identical across batch sizes.

* selection workload: fp32 logits [512 x 8 rows, 152064], T = 0.7 and T = 0,
  peaked / near-tie / exact-tie rows, drafts wrong at 20% of positions;
* Llama-3-8B-shaped layer + LM head (d 4096, 32/8 heads, FFN 14336, vocab
  128256), M in {1, 8, 32, 64, 128, 256} rows with 4096 cached positions each;
* verifier sweep on those shapes: N x K windows with lognormal contexts.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, same_bits
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth
from invariant_verify_gb300.verifier import DecoderVerifier, make_window

pytestmark = pytest.mark.gpu
SEED = synth.PHILOX_SEED


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_verify_gb300 import build
    build.build()
    yield
    assert B.biv_device_error() == 0


# ------------------------------------------------------------- selection
@pytest.mark.parametrize("T,exact_ties", [(0.7, False), (0.0, False), (0.0, True)])
def test_selection_full_size_bit_exact(T, exact_ties):
    cfg = synth.SELECT
    x, kind = synth.select_logits(cfg, exact_ties=exact_ties)
    R = cfg.R
    req = torch.arange(cfg.requests, dtype=torch.int32).repeat_interleave(cfg.K) * 7 + 3
    p0 = torch.randint(100, 30000, (cfg.requests,), generator=synth.generator(91), dtype=torch.int64)
    pos = (p0.repeat_interleave(cfg.K) + torch.arange(cfg.K).repeat(cfg.requests)).to(torch.int32)
    xd = x.cuda()
    tok = torch.empty(R, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(xd, req.cuda(), pos.cuda(), SEED, T, tok)
    # the workspace entry (flat rows to the unit kernel): the same tokens
    ws = torch.empty(B.biv_gumbel_argmax_workspace_size(R, cfg.vocab), dtype=torch.uint8, device="cuda")
    tok_ws = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax_ws(xd, req.cuda(), pos.cuda(), SEED, T, tok_ws, ws)
    torch.cuda.synchronize()
    del xd, ws
    ref = oracle.gumbel_argmax(x, req, pos, SEED, T)
    assert np.array_equal(tok.cpu().numpy(), ref)
    assert torch.equal(tok_ws, tok)
    # drafts = targets with 20% random ids; accept lengths and rollback points bit-exact
    mask, ids = synth.draft_errors((R,), cfg.draft_err, cfg.vocab, seed=92)
    draft = synth.apply_draft_errors(torch.from_numpy(ref), mask, ids)
    p0i = p0.to(torch.int32)
    L = torch.empty(cfg.requests, dtype=torch.int32, device="cuda")
    nl = torch.empty(cfg.requests, dtype=torch.int32, device="cuda")
    B.biv_verify_accept(tok, draft.cuda(), p0i.cuda(), cfg.requests, cfg.K, L, nl)
    rL, rnl = oracle.verify_accept(ref, draft, p0i, cfg.requests, cfg.K)
    assert np.array_equal(L.cpu().numpy(), rL) and np.array_equal(nl.cpu().numpy(), rnl)
    if exact_ties:
        # every tie row really tied: greedy picks the lower of the two indices
        tie_rows = np.nonzero(kind.numpy() == 1)[0]
        xr = x[tie_rows].numpy()
        top = xr.max(axis=1)
        assert np.array_equal(ref[tie_rows], np.argmax(xr == top[:, None], axis=1))


# ------------------------------------------------- Llama-3-8B-shaped layer
M_SWEEP = (1, 8, 32, 64, 128, 256)


@pytest.fixture(scope="module")
def llama():
    cfg = synth.LLAMA8B
    M = max(M_SWEEP)
    w = synth.decoder_weights_device(cfg)
    ctx = torch.full((M,), 4096, dtype=torch.int32)
    max_len = 4096 + 64
    caches = synth.kv_cache_device(M, cfg.Hkv, max_len, cfg.hd, ctx, seed=33, layers=cfg.layers)
    toks = torch.randint(0, cfg.vocab, (M,), generator=synth.generator(34), dtype=torch.int64).to(torch.int32)
    req = torch.arange(M, dtype=torch.int32) * 13 + 5
    return cfg, w, caches, ctx, max_len, toks, req


def test_llama_layer_rows_bitwise_across_M(llama):
    cfg, w, caches, ctx, max_len, toks, req = llama
    M = max(M_SWEEP)
    full = DecoderVerifier(cfg, w, caches, M, max_len, M, 1)
    full.step(make_window(M, 1, toks, ctx, req, toks))
    torch.cuda.synchronize()
    H, Lg, T = full.hidden.clone(), full.logits.clone(), full.target.clone()
    del full
    for m in M_SWEEP[:-1]:
        v = DecoderVerifier(cfg, w, caches, M, max_len, m, 1)
        v.step(make_window(m, 1, toks[:m], ctx[:m], req[:m], toks[:m]))
        torch.cuda.synchronize()
        assert same_bits(v.hidden, H[:m]) and same_bits(v.logits, Lg[:m]) and same_bits(v.target, T[:m]), m
        del v


def _sample_pairs(M, N, n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, M, n), rng.integers(0, N, n)


def sampled_stage_parity(cfg, w, ver, win, rows, seed=0):
    """Every stage of one traced Llama-3-8B-shaped step against the oracle on
    sampled elements, each stage fed the GPU's own input for it (so the
    per-kernel tolerance applies): RMSNorm (all rows), the QKV, Wo, gate/up +
    SwiGLU, down and LM-head GEMMs on 256-512 sampled (row, column) pairs,
    RoPE and attention on the given rows (one head each, spread over the
    heads), and the selection bit-exact on the GPU's logits."""
    M = ver.W
    Hq, Hkv, hd = cfg.Hq, cfg.Hkv, cfg.hd
    tr = {}
    ver.forward(win, trace=tr)
    ver.lm_head(win)
    ver.select_and_accept(win)
    torch.cuda.synchronize()
    cpu = {k: v.cpu() for k, v in tr.items() if not k.endswith("kc") and not k.endswith("vc")}
    pos = win.row_pos.cpu().numpy()

    def gemm_check(a, wname, out, s, what):
        m, n = _sample_pairs(a.shape[0], out.shape[1], 512, seed + s)
        ref = oracle.gemm_sampled(a, w[wname].cpu(), m, n)
        got = out.float().numpy()[m, n]
        assert_close(torch.from_numpy(got), ref, what=what)

    ones = np.ones(cfg.d)
    assert_close(cpu["l0.h_attn"], oracle.rmsnorm(cpu["x_in"], ones, cfg.eps), what="rmsnorm")
    gemm_check(cpu["l0.h_attn"], "l0.wqkv", cpu["l0.qkv"], 1, "qkv")
    rows = np.asarray(rows)
    R = rows.size
    qkv = oracle.from_bf16(cpu["l0.qkv"][rows])
    assert_close(cpu["l0.q"][rows], oracle.rope(qkv[:, :Hq * hd].reshape(R, Hq, hd), pos[rows], cfg.rope_theta),
                 what="rope")
    # attention on sampled (row, head) pairs, against the cache the window wrote
    kc, vc = tr["l0.kc"], tr["l0.vc"]
    slots = win.row_slot.cpu().numpy()[rows]
    kc_s = kc[torch.as_tensor(slots).cuda()].cpu()
    vc_s = vc[torch.as_tensor(slots).cuda()].cpu()
    heads = (np.arange(R) * 7 + 5 * (seed % 3)) % Hq
    ref = oracle.attention_sampled(cpu["l0.q"][rows], kc_s, vc_s, np.arange(R), pos[rows], np.arange(R), heads)
    got = cpu["l0.o"][rows, heads].float()
    assert_close(got, ref, what="attention")
    gemm_check(cpu["l0.o"].view(M, Hq * hd), "l0.wo", cpu["l0.attn_proj"], 2, "wo")
    # gate/up + SwiGLU on sampled (row, i): act = silu(bf16(g)) * bf16(u)
    F = cfg.ffn
    m, i = _sample_pairs(M, F, 256, seed + 3)
    wgu = w["l0.wgu"].cpu()
    g = oracle.round_bf16(oracle.gemm_sampled(cpu["l0.h_ffn"], wgu, m, i))
    u = oracle.round_bf16(oracle.gemm_sampled(cpu["l0.h_ffn"], wgu, m, F + i))
    ref = oracle.silu_mul(np.stack([g, u], axis=1))[:, 0]
    assert_close(torch.from_numpy(cpu["l0.act"].float().numpy()[m, i]), ref, what="gate/up + swiglu")
    gemm_check(cpu["l0.act"], "l0.wdown", cpu["l0.down"], 4, "down")
    gemm_check(cpu["hidden"], "lm_head", ver.logits.cpu(), 5, "lm head")
    tgt = oracle.gumbel_argmax(ver.logits.cpu(), win.row_req.cpu(), pos, SEED, cfg.temperature)
    assert np.array_equal(ver.target.cpu().numpy(), tgt)


def test_llama_layer_sampled_parity(llama):
    cfg, w, caches, ctx, max_len, toks, req = llama
    M = max(M_SWEEP)
    ver = DecoderVerifier(cfg, w, caches, M, max_len, M, 1)
    win = make_window(M, 1, toks, ctx, req, toks)
    sampled_stage_parity(cfg, w, ver, win, [0, 17, 101, 255])


# ------------------------------------------------------- verifier sweep
@pytest.mark.parametrize("N,K", [(8, 4), (32, 8), (64, 16)])
def test_sweep_window_accept_and_invariance(N, K):
    cfg = synth.SWEEP
    w = synth.decoder_weights_device(cfg)
    ctx = synth.context_lengths(cfg, N, seed=40 + N)
    max_len = int(ctx.max()) + K + 16
    caches = synth.kv_cache_device(N, cfg.Hkv, max_len, cfg.hd, ctx, seed=41 + N, layers=cfg.layers)
    W = N * K
    ver = DecoderVerifier(cfg, w, caches, N, max_len, W, K)
    req = torch.arange(N, dtype=torch.int32) * 31 + 1
    last = torch.randint(0, cfg.vocab, (N,), generator=synth.generator(43), dtype=torch.int64).to(torch.int32)
    mask, ids = synth.draft_errors((N, K), cfg.draft_err, cfg.vocab, seed=44)
    drafts = torch.zeros(N, K, dtype=torch.int32)
    for j in range(K):    # drafts that disagree with the verifier at 20% of positions
        tokens = torch.cat([last[:, None], drafts[:, :-1]], dim=1)
        ver.step(make_window(N, K, tokens.reshape(-1), ctx, req, drafts.reshape(-1)))
        drafts[:, j] = torch.where(mask[:, j], ids[:, j], ver.target.view(N, K)[:, j].cpu())
    tokens = torch.cat([last[:, None], drafts[:, :-1]], dim=1)
    win = make_window(N, K, tokens.reshape(-1), ctx, req, drafts.reshape(-1))
    ver.step(win)
    torch.cuda.synchronize()
    tgt = ver.target.cpu().numpy()
    if W == 1024:
        ref = oracle.gumbel_argmax(ver.logits.cpu(), win.row_req.cpu(), win.row_pos.cpu(), SEED, cfg.temperature)
        assert np.array_equal(tgt, ref)
    rL, rnl = oracle.verify_accept(tgt, drafts.reshape(-1), ctx, N, K)
    assert np.array_equal(ver.accept_len.cpu().numpy(), rL) and np.array_equal(ver.new_len.cpu().numpy(), rnl)
    # The targets seen while the drafts were built equal the final ones (rows
    # are invariant to the drafts after them), so every request breaks exactly
    # at its first deliberately wrong draft.
    eff = mask.numpy() & (ids.numpy() != tgt.reshape(N, K))
    assert np.array_equal(rL, np.where(eff.any(axis=1), eff.argmax(axis=1) + 1, K))
    if W == 1024:
        # dense stages of the largest window on sampled elements, in the
        # configuration the benchmark times (CTA-pair GEMM tiles, G*K = 64-row
        # attention tiles over contexts up to 8192)
        sampled_stage_parity(cfg, w, ver, win, [0, 17, 333, 600, 777, 1023], seed=10)
    # rows of the first and last request computed alone give the same bits
    for r in (0, N - 1):
        sl = slice(r * K, (r + 1) * K)
        one = DecoderVerifier(cfg, w, caches, N, max_len, K, K)
        one.kc, one.vc = ver.kc, ver.vc
        wi = make_window(1, K, tokens[r], ctx[r:r + 1], req[r:r + 1], drafts[r])
        wi.row_slot.fill_(r)
        one.step(wi)
        assert same_bits(one.hidden, ver.hidden[sl]) and same_bits(one.logits, ver.logits[sl])
        assert same_bits(one.target, ver.target[sl])
