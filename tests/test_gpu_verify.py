"""End-to-end verify steps on the GPU through the C ABI.

* Tiny workload (RMSNorm d=256 -> LM head 2048 -> select T=1 -> accept,
  N=4 x K=4): parity with the oracle and bitwise batch invariance at
  W in {1, 2, 4, 8, 16}.
* 2-layer decoder verifier (d=1024, 8/2 heads, FFN 2816, vocab 32000,
  N=8 x K=8, T=0.7): logits within tolerance of the oracle composition,
  tokens and accept lengths bit-exact against the oracle's selection of the
  same logits, every row bitwise identical when recomputed alone or in a
  permuted window, and drafter invariance of the Decode-Verify-Rollback loop.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.model import OracleDecoder
from gpu_util import assert_close, check_end_to_end, dev, e2e_logit_envelope, same_bits
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth
from invariant_verify_gb300.verifier import DecoderVerifier, Window, make_window

pytestmark = pytest.mark.gpu
SEED = 0x1234_5678_9ABC_DEF0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_verify_gb300 import build
    build.build()
    yield
    assert B.biv_device_error() == 0


def i32(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32).cuda()


# ------------------------------------------------------------ tiny workload
def tiny_step(h, gain, lm, row_req, row_pos, T):
    W, d = h.shape
    hn = torch.empty_like(h)
    B.biv_rmsnorm(h, gain, hn, synth.TINY.eps)
    logits = torch.empty(W, lm.shape[0], dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(hn, lm, logits)
    tok = torch.empty(W, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(logits, row_req, row_pos, SEED, T, tok)
    return hn, logits, tok


def test_tiny_parity_and_invariance():
    cfg = synth.TINY
    inp = synth.tiny_inputs(cfg)
    N, K = cfg.N, cfg.K
    W = N * K
    _, row_req, row_pos = synth.request_window(N, K, inp["p0"], inp["req_ids"])
    h, gain, lm = dev(inp["h"]), dev(inp["gain"]), dev(inp["lm_head"])
    hn, logits, tok = tiny_step(h, gain, lm, i32(row_req), i32(row_pos), cfg.temperature)
    # parity: each stage against the oracle on the same inputs
    assert_close(hn, oracle.rmsnorm(inp["h"], inp["gain"], cfg.eps), what="tiny rmsnorm")
    assert_close(logits, oracle.gemm(hn.cpu(), inp["lm_head"]), what="tiny logits")
    ref_tok = oracle.gumbel_argmax(logits.cpu(), row_req, row_pos, SEED, cfg.temperature)
    assert np.array_equal(tok.cpu().numpy(), ref_tok)
    # drafts = target tokens with 25% replaced; accept lengths bit-exact
    mask, ids = synth.draft_errors((W,), cfg.draft_err, cfg.vocab, seed=7)
    draft = synth.apply_draft_errors(torch.tensor(ref_tok), mask, ids)
    L = torch.empty(N, dtype=torch.int32, device="cuda")
    nl = torch.empty(N, dtype=torch.int32, device="cuda")
    B.biv_verify_accept(tok, dev(draft), dev(inp["p0"]), N, K, L, nl)
    rL, rnl = oracle.verify_accept(ref_tok, draft, inp["p0"], N, K)
    assert np.array_equal(L.cpu().numpy(), rL) and np.array_equal(nl.cpu().numpy(), rnl)
    # batch invariance at W in {1, 2, 4, 8, 16}, every offset
    for w in cfg.invariance_W:
        for start in range(0, W, w):
            sl = slice(start, start + w)
            hn2, lg2, tk2 = tiny_step(h[sl].contiguous(), gain, lm, i32(row_req[sl]), i32(row_pos[sl]),
                                      cfg.temperature)
            assert same_bits(hn2, hn[sl]) and same_bits(lg2, logits[sl]) and same_bits(tk2, tok[sl]), (w, start)


# ---------------------------------------------------- 2-layer decoder verifier
def decoder_setup(cfg=synth.DECODER2):
    w = synth.decoder_weights(cfg)
    ctx = synth.context_lengths(cfg, cfg.N, seed=cfg.seed + 100)
    max_len = int(ctx.max()) + 64
    caches = synth.kv_cache(cfg.N, cfg.Hkv, max_len, cfg.hd, ctx, seed=cfg.seed + 200, layers=cfg.layers)
    return w, caches, ctx, max_len


@pytest.fixture(scope="module")
def dec2():
    return decoder_setup()


def _window(cfg, ctx, tokens, draft, p0=None):
    p0 = ctx if p0 is None else p0
    return make_window(cfg.N, cfg.K, tokens, p0, torch.arange(cfg.N) * 1000 + 17, draft)


def _cpu(t):
    return t.detach().cpu()


def test_decoder_stagewise_parity(dec2):
    """Every kernel of the composed step against the oracle, each fed the
    GPU's own inputs for that stage (so the tolerance is the per-kernel one)."""
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    W, Hq, Hkv, hd = cfg.W, cfg.Hq, cfg.Hkv, cfg.hd
    toks = torch.randint(0, cfg.vocab, (W,), generator=synth.generator(50), dtype=torch.int64).to(torch.int32)
    win = _window(cfg, ctx, toks, toks)
    ver = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, cfg.K)
    tr = {}
    ver.forward(win, trace=tr)
    ver.lm_head(win)
    ver.select_and_accept(win)
    torch.cuda.synchronize()
    slot, pos = win.row_slot.cpu().numpy(), win.row_pos.cpu().numpy()
    ones = np.ones(cfg.d)
    assert torch.equal(_cpu(tr["x_in"]), w["embed"][toks.long()])
    x = tr["x_in"]
    for l in range(cfg.layers):
        assert_close(tr[f"l{l}.h_attn"], oracle.rmsnorm(_cpu(x), ones, cfg.eps), what=f"l{l} rmsnorm")
        assert_close(tr[f"l{l}.qkv"], oracle.gemm(_cpu(tr[f"l{l}.h_attn"]), w[f"l{l}.wqkv"]), what=f"l{l} qkv")
        qkv = oracle.from_bf16(_cpu(tr[f"l{l}.qkv"]))
        assert_close(tr[f"l{l}.q"], oracle.rope(qkv[:, :Hq * hd].reshape(W, Hq, hd), pos, cfg.rope_theta),
                     what=f"l{l} rope q")
        # KV overwrite: the window rows hold the rotated k and the raw v, every other row is untouched
        k_ref = oracle.rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(W, Hkv, hd), pos, cfg.rope_theta)
        kc_gpu = _cpu(tr[f"l{l}.kc"])
        assert_close(kc_gpu[slot, :, pos].float(), k_ref, what=f"l{l} rope k in cache")
        kc = oracle._np(caches[l][0]).copy(); vc = oracle._np(caches[l][1]).copy()
        vnew = oracle._np(_cpu(tr[f"l{l}.qkv"])[:, (Hq + Hkv) * hd:].contiguous()).reshape(W, Hkv, hd)
        oracle.kv_overwrite(kc, vc, oracle._np(kc_gpu[slot, :, pos].contiguous()), vnew, slot, pos)
        assert np.array_equal(oracle._np(kc_gpu), kc)
        assert np.array_equal(oracle._np(_cpu(tr[f"l{l}.vc"])), vc)
        assert_close(tr[f"l{l}.o"], oracle.attention(_cpu(tr[f"l{l}.q"]), kc, vc, slot, pos), what=f"l{l} attn")
        assert_close(tr[f"l{l}.attn_proj"], oracle.gemm(_cpu(tr[f"l{l}.o"]).view(W, Hq * hd), w[f"l{l}.wo"]),
                     what=f"l{l} wo")
        assert_close(tr[f"l{l}.x_mid"], oracle.from_bf16(_cpu(x)) + oracle.from_bf16(_cpu(tr[f"l{l}.attn_proj"])),
                     what=f"l{l} residual")
        assert_close(tr[f"l{l}.h_ffn"], oracle.rmsnorm(_cpu(tr[f"l{l}.x_mid"]), ones, cfg.eps), what=f"l{l} norm2")
        gu = oracle.round_bf16(oracle.gemm(_cpu(tr[f"l{l}.h_ffn"]), w[f"l{l}.wgu"]))
        assert_close(tr[f"l{l}.act"], oracle.silu_mul(gu), what=f"l{l} gate/up + swiglu")
        assert_close(tr[f"l{l}.down"], oracle.gemm(_cpu(tr[f"l{l}.act"]), w[f"l{l}.wdown"]), what=f"l{l} down")
        assert_close(tr[f"l{l}.x_out"], oracle.from_bf16(_cpu(tr[f"l{l}.x_mid"])) +
                     oracle.from_bf16(_cpu(tr[f"l{l}.down"])), what=f"l{l} residual 2")
        x = tr[f"l{l}.x_out"]
    assert_close(tr["hidden"], oracle.rmsnorm(_cpu(x), ones, cfg.eps), what="final norm")
    assert_close(ver.logits, oracle.gemm(_cpu(tr["hidden"]), w["lm_head"]), what="lm head")
    # selection and accept: bit-exact against the oracle on the GPU's logits
    tgt = oracle.gumbel_argmax(_cpu(ver.logits), _cpu(win.row_req), pos, SEED, cfg.temperature)
    assert np.array_equal(ver.target.cpu().numpy(), tgt)
    rL, rnl = oracle.verify_accept(tgt, toks.numpy(), ctx.numpy(), cfg.N, cfg.K)
    assert np.array_equal(ver.accept_len.cpu().numpy(), rL)
    assert np.array_equal(ver.new_len.cpu().numpy(), rnl)


def test_decoder_end_to_end_against_oracle(dec2):
    """The whole step against the oracle's own composition (no GPU value fed
    back): logits within the rounding-drift envelope of gpu_util (derived
    from the oracle, row by row), and every token that differs from the
    oracle's explained by a key gap the logit drift bridges."""
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    W = cfg.W
    toks = torch.randint(0, cfg.vocab, (W,), generator=synth.generator(50), dtype=torch.int64).to(torch.int32)
    win = _window(cfg, ctx, toks, toks)
    ver = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, cfg.K)
    ver.step(win)
    torch.cuda.synchronize()
    orc = OracleDecoder(cfg, w, caches, cfg.N, max_len)
    slot, pos = win.row_slot.cpu().numpy(), win.row_pos.cpu().numpy()
    ref, tol = e2e_logit_envelope(orc, toks.numpy(), slot, pos)
    agree = check_end_to_end(ver.logits.cpu().numpy(), ver.target.cpu().numpy(), ref, tol, win.row_req.cpu(),
                             pos, SEED, cfg.temperature, what="2-layer decoder")
    print(f"end-to-end: envelope {tol.min():.4f}..{tol.max():.4f}, token agreement {agree}/{W}")


def test_decoder_rows_bitwise_invariant(dec2):
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    W = cfg.W
    toks = torch.randint(0, cfg.vocab, (W,), generator=synth.generator(51), dtype=torch.int64).to(torch.int32)
    full = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, cfg.K)
    win = _window(cfg, ctx, toks, toks)
    full.step(win)
    torch.cuda.synchronize()
    H, Lg, Tg = full.hidden.clone(), full.logits.clone(), full.target.clone()
    # every row alone (W = 1) against the cache the window wrote
    one = DecoderVerifier(cfg, w, caches, cfg.N, max_len, 1, 1)
    one.kc, one.vc = full.kc, full.vc
    for r in range(W):
        sl = slice(r, r + 1)
        wi = Window(win.tokens[sl], win.row_slot[sl], win.row_req[sl], win.row_pos[sl], win.draft[sl],
                    win.row_pos[sl].clone())
        one.step(wi)
        assert same_bits(one.hidden[0], H[r]) and same_bits(one.logits[0], Lg[r]) and same_bits(one.target[0], Tg[r]), r
    # a permuted window (groups of one row)
    perm = torch.randperm(W, generator=synth.generator(52)).cuda()
    pv = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, 1)
    pv.kc, pv.vc = full.kc, full.vc
    pw = Window(win.tokens[perm].contiguous(), win.row_slot[perm].contiguous(), win.row_req[perm].contiguous(),
                win.row_pos[perm].contiguous(), win.draft[perm].contiguous(), win.row_pos[perm].contiguous())
    pv.step(pw)
    assert same_bits(pv.hidden, H[perm]) and same_bits(pv.logits, Lg[perm]) and same_bits(pv.target, Tg[perm])
    # a CUDA-graph replay gives the same bits
    g = full.capture(win)
    g.replay()
    torch.cuda.synchronize()
    assert same_bits(full.logits, Lg) and same_bits(full.target, Tg)


def test_end_to_end_graph_with_host_buffers(dec2):
    """The end-to-end path: window inputs copied from one pinned host buffer,
    the step, results copied back into one pinned host buffer, all in one
    graph -- the same tokens, accept lengths and rollback points as a plain
    step, replay after replay, and a second window through the same graph."""
    from invariant_verify_gb300.verifier import PackedWindow, capture_e2e
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    W = cfg.W
    g = synth.generator(61)
    wins = []
    for _ in range(2):
        toks = torch.randint(0, cfg.vocab, (W,), generator=g, dtype=torch.int64).to(torch.int32)
        drafts = torch.randint(0, cfg.vocab, (W,), generator=g, dtype=torch.int64).to(torch.int32)
        wins.append(_window(cfg, ctx, toks, drafts))
    refs = []
    for wi in wins:
        ver = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, cfg.K)
        ver.step(wi)
        torch.cuda.synchronize()
        refs.append(ver.results.cpu().clone())
    ver = DecoderVerifier(cfg, w, caches, cfg.N, max_len, W, cfg.K)
    pw = PackedWindow(cfg.N, cfg.K)
    host_out = torch.empty_like(ver.results, device="cpu").pin_memory()
    pw.set(wins[0])
    graph = capture_e2e(ver, pw, host_out)
    for wi, ref in ((wins[0], refs[0]), (wins[1], refs[1]), (wins[0], refs[0])):
        pw.set(wi)
        host_out.fill_(-1)
        graph.replay()
        torch.cuda.current_stream().synchronize()
        assert torch.equal(host_out, ref)


def test_fast_path_kv_is_overwritten(dec2):
    # Perturb the window's cache rows (a stale fast path) before verifying:
    # the verifier overwrites them and the result equals a clean run.
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    toks = torch.randint(0, cfg.vocab, (cfg.W,), generator=synth.generator(53), dtype=torch.int64).to(torch.int32)
    win = _window(cfg, ctx, toks, toks)
    clean = DecoderVerifier(cfg, w, caches, cfg.N, max_len, cfg.W, cfg.K)
    clean.step(win)
    dirty = DecoderVerifier(cfg, w, caches, cfg.N, max_len, cfg.W, cfg.K)
    for l in range(cfg.layers):
        for r in range(cfg.N):
            p = int(ctx[r])
            dirty.kc[l][r, :, p:p + cfg.K] += 0.5
            dirty.vc[l][r, :, p:p + cfg.K] -= 0.25
    dirty.step(win)
    torch.cuda.synchronize()
    assert same_bits(dirty.logits, clean.logits) and same_bits(dirty.target, clean.target)


def gpu_dvr_decode(cfg, w, caches, ctx, max_len, n_tokens, K, drafter, first):
    """Decode-Verify-Rollback on the GPU: returns the committed streams."""
    N = cfg.N
    ver = DecoderVerifier(cfg, w, caches, N, max_len, N * K, K)
    last = list(first)
    pos = [int(c) for c in ctx]
    streams = [[] for _ in range(N)]
    req = torch.arange(N) * 1000 + 17
    while min(len(s) for s in streams) < n_tokens:
        drafts = np.array([drafter(r, streams[r], K) for r in range(N)], np.int32).reshape(N, K)
        tokens = np.empty((N, K), np.int32)
        tokens[:, 0] = last
        tokens[:, 1:] = drafts[:, :-1]
        win = make_window(N, K, tokens.reshape(-1), pos, req, drafts.reshape(-1))
        ver.step(win)
        L = ver.accept_len.cpu().numpy()
        tgt = ver.target.cpu().numpy().reshape(N, K)
        for r in range(N):
            streams[r].extend(int(t) for t in tgt[r, :L[r]])
            last[r] = int(tgt[r, L[r] - 1])
            pos[r] += int(L[r])
    return [s[:n_tokens] for s in streams]


def test_drafter_invariance_on_gpu(dec2):
    cfg = synth.DECODER2
    w, caches, ctx, max_len = dec2
    n_tokens = 24
    first = list(range(100, 100 + cfg.N))
    rng = np.random.default_rng(9)
    none = gpu_dvr_decode(cfg, w, caches, ctx, max_len, n_tokens, 1, lambda r, h, K: [0] * K, first)
    rand = gpu_dvr_decode(cfg, w, caches, ctx, max_len, n_tokens, 8,
                          lambda r, h, K: list(rng.integers(0, cfg.vocab, K)), first)

    def perfect(r, h, K):
        fut = none[r][len(h):len(h) + K]
        return fut + [0] * (K - len(fut))

    perf = gpu_dvr_decode(cfg, w, caches, ctx, max_len, n_tokens, 8, perfect, first)

    def noisy(r, h, K):   # 30% random-token error rate per position
        d = perfect(r, h, K)
        return [int(rng.integers(0, cfg.vocab)) if rng.random() < cfg.draft_err else t for t in d]

    mixed = gpu_dvr_decode(cfg, w, caches, ctx, max_len, n_tokens, 8, noisy, first)
    assert none == rand == perf == mixed
