"""GPU parity of the Gumbel top-k selection and the n-gram lookup drafter
against the oracle (bit-exact: both produce integers), and the drafter-
invariance of a decode loop that uses the n-gram drafter."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import same_bits
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


# ---------------------------------------------------------------- top-k
@pytest.mark.parametrize("R,V,T,k,std", [
    (16, 2048, 1.0, 8, 1.0), (64, 32000, 0.7, 4, 0.64), (9, 152064, 0.7, 16, 3.0), (5, 8, 1.0, 8, 1.0),
    (33, 4100, 0.0, 64, 1.0), (7, 1000, 2.0, 1, 0.5), (12, 256, 1e-3, 32, 1.0)])
def test_topk_bit_exact(R, V, T, k, std):
    g = synth.generator(R * 7 + V + k)
    x = torch.randn(R, V, generator=g) * std
    if V >= 300:
        x[0, 100] = x[0, 250] = x[0].max() + 1.0          # exact tie at the top
        x[1, 7] = float("nan")
    req = torch.randint(0, 2 ** 31 - 1, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    pos = torch.randint(0, 9000, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    out = torch.full((R, k), -5, dtype=torch.int32, device="cuda")
    B.biv_gumbel_topk(x.cuda(), req.cuda(), pos.cuda(), SEED, T, out)
    ref = oracle.gumbel_topk(x, req, pos, SEED, T, k)
    assert np.array_equal(out.cpu().numpy(), ref)
    tok = torch.empty(R, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(x.cuda(), req.cuda(), pos.cuda(), SEED, T, tok)
    assert torch.equal(tok.cpu(), out[:, 0].cpu())


# --------------------------------------------------------------- n-gram
def _histories(N, ld, alphabet, seed):
    rng = np.random.default_rng(seed)
    h = rng.integers(0, alphabet, (N, ld)).astype(np.int32)
    lens = rng.integers(0, ld + 1, N).astype(np.int32)
    # some periodic rows, some with a planted long repeat
    for r in range(0, N, 5):
        period = 2 + r % 7
        h[r] = np.tile(h[r, :period], ld // period + 1)[:ld]
    for r in range(1, N, 5):
        L = int(lens[r])
        if L > 40:
            h[r, L - 12:L] = h[r, 10:22]
    lens[:3] = [0, 1, 2]
    return h, lens


@pytest.mark.parametrize("N,ld,alphabet,n_max,n_min,K", [
    (64, 512, 6, 4, 1, 8), (32, 8192, 50, 8, 2, 16), (7, 100, 3, 3, 3, 5), (128, 2048, 1000, 5, 1, 4)])
def test_ngram_draft_bit_exact(N, ld, alphabet, n_max, n_min, K):
    h, lens = _histories(N, ld, alphabet, seed=N + ld)
    d = torch.full((N, K), -9, dtype=torch.int32, device="cuda")
    src = torch.full((N,), -9, dtype=torch.int32, device="cuda")
    B.biv_ngram_draft(torch.from_numpy(h).cuda(), torch.from_numpy(lens).cuda(), n_max, n_min, d, src)
    rd, rsrc = oracle.ngram_draft(h, lens, n_max, n_min, K)
    assert np.array_equal(src.cpu().numpy(), rsrc)
    assert np.array_equal(d.cpu().numpy(), rd)


def test_ngram_drafter_decode_is_drafter_invariant():
    """Decode 24 tokens per request with n-gram drafts (K = 6) and with no
    drafts (K = 1): the committed streams are identical (coupled selection and
    batch-invariant rows), whatever the drafter proposes."""
    cfg = synth.DECODER2
    N, K, steps_tokens = 4, 6, 24
    w = synth.decoder_weights_device(cfg)
    ctx0 = 64
    max_len = ctx0 + steps_tokens + 2 * K + 8
    caches = synth.kv_cache_device(N, cfg.Hkv, max_len, cfg.hd, torch.full((N,), ctx0, dtype=torch.int32),
                                   seed=71, layers=cfg.layers)
    req = torch.arange(N, dtype=torch.int32) * 5 + 2
    g = synth.generator(72)
    # repetitive history so the n-gram drafter finds matches
    base = torch.randint(0, cfg.vocab, (N, 8), generator=g, dtype=torch.int64).to(torch.int32)
    hist0 = base.repeat(1, ctx0 // 8)

    def decode(k_rows, use_ngram):
        ver = DecoderVerifier(cfg, w, [(a.clone(), b.clone()) for a, b in caches], N, max_len, N * k_rows, k_rows)
        hist = torch.zeros(N, max_len, dtype=torch.int32, device="cuda")
        hist[:, :ctx0] = hist0.cuda()
        lens = torch.full((N,), ctx0, dtype=torch.int32)
        drafts = torch.empty(N, k_rows, dtype=torch.int32, device="cuda")
        src = torch.empty(N, dtype=torch.int32, device="cuda")
        while int(lens.min()) < ctx0 + steps_tokens:
            if use_ngram:
                B.biv_ngram_draft(hist, lens.cuda(), 4, 1, drafts, src)
                d = drafts.cpu()
            else:
                d = torch.zeros(N, k_rows, dtype=torch.int32)
            last = torch.stack([hist[r, int(lens[r]) - 1].cpu() for r in range(N)])
            tokens = torch.cat([last[:, None], d[:, :-1]], dim=1)
            p0 = lens - 1                     # position of the last committed token
            win = make_window(N, k_rows, tokens.reshape(-1), p0, req, d.reshape(-1))
            ver.step(win)
            L = ver.accept_len.cpu()
            tgt = ver.target.view(N, k_rows).cpu()
            for r in range(N):
                n = int(L[r])
                hist[r, int(lens[r]):int(lens[r]) + n] = tgt[r, :n].cuda()
                lens[r] += n
        return [hist[r, ctx0:ctx0 + steps_tokens].cpu() for r in range(N)]

    ref = decode(1, False)
    got = decode(K, True)
    for r in range(N):
        assert torch.equal(ref[r], got[r]), r
