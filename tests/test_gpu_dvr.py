"""Decode-Verify-Rollback with the batch-variant fast path as the drafter
(§8(f) f2).  The fast path is PyTorch on cuBLAS with its own KV cache; the
verifier is the library's batch-invariant step.  Checked: the committed
streams equal those of verifying without any drafter, bit for bit (coupled
selection: the drafter only changes how many tokens a round commits), the
fast path's cache holds the verifier's K/V for every committed position, and
the fast path's divergence rate (drafts the verifier rejects) is reported."""
import pytest
import torch

from gpu_util import same_bits
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth
from invariant_verify_gb300.fastpath import FastPathDecoder, dvr_generate
from invariant_verify_gb300.verifier import DecoderVerifier

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


@pytest.mark.parametrize("K", [4, 8])
def test_dvr_with_fast_path_commits_the_verifier_stream(K):
    cfg = synth.DECODER2
    N, n_tokens = 6, 40
    w = synth.decoder_weights_device(cfg)
    ctx = synth.context_lengths(cfg, N, seed=90 + K)
    max_len = int(ctx.max()) + n_tokens + 2 * K + 8
    caches = synth.kv_cache_device(N, cfg.Hkv, max_len, cfg.hd, ctx, seed=91, layers=cfg.layers)
    req = torch.arange(N, dtype=torch.int32) * 37 + 11
    last = torch.randint(0, cfg.vocab, (N,), generator=synth.generator(92), dtype=torch.int64).to(torch.int32)
    p0 = (ctx - 1).to(torch.int32)

    def fresh(k_rows):
        return DecoderVerifier(cfg, w, [(a.clone(), b.clone()) for a, b in caches], N, max_len, N * k_rows, k_rows)

    ref, _ = dvr_generate(fresh(1), None, last, p0, req, n_tokens)
    ver = fresh(K)
    fast = FastPathDecoder(cfg, w, caches, SEED)
    got, st = dvr_generate(ver, fast, last, p0, req, n_tokens)
    for r in range(N):
        assert torch.equal(ref[r], got[r]), r
    print(f"K={K}: rounds {st.rounds}, drafted {st.drafted}, accepted {st.accepted}, "
          f"divergence rate {st.divergence_rate:.4f}, committed/round {st.committed / st.rounds / N:.2f}")
    # the fast path is a good drafter (same model, different rounding): most drafts are accepted
    assert st.divergence_rate < 0.25
    # rollback + overwrite: every committed position holds the verifier's K/V in the fast cache
    for r in range(N):
        a, b = int(p0[r]), int(p0[r]) + n_tokens
        for l in range(cfg.layers):
            assert same_bits(fast.kc[l][r, :, a:b], ver.kc[l][r, :, a:b])
            assert same_bits(fast.vc[l][r, :, a:b], ver.vc[l][r, :, a:b])


def test_fast_path_is_batch_variant_where_the_verifier_is_not():
    """The fast path's logits for the same rows change bits with the batch
    size (cuBLAS is free to pick another reduction); the verifier's do not."""
    cfg = synth.DECODER2
    w = synth.decoder_weights_device(cfg)
    g = synth.generator(95)
    h = synth.bf16_normal((256, cfg.d), 1.0, g).cuda()
    fast_small = h[:3] @ w["lm_head"].t()
    fast_big = (h @ w["lm_head"].t())[:3]
    ours_small = torch.empty(3, cfg.vocab, dtype=torch.float32, device="cuda")
    ours_big = torch.empty(256, cfg.vocab, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(h[:3].contiguous(), w["lm_head"], ours_small)
    B.biv_gemm_nosplitk(h, w["lm_head"], ours_big)
    assert same_bits(ours_small, ours_big[:3])
    print("cuBLAS rows identical across batch sizes:", bool(torch.equal(fast_small, fast_big)))
