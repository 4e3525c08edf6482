"""Deterministic prefill (§8(f) f3): the prompt runs as one window of one
request (rows at positions 0..P-1, no split-K, fixed-split causal attention).
Because every row is computed the same way whatever else is in the window,
the prefill writes exactly the KV cache, and selects exactly the tokens, that
feeding the prompt one token per step does -- checked bitwise -- and it agrees
with the fp64 oracle's composition within the rounding-drift envelope (row
by row, derived from the oracle; see gpu_util)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_end_to_end, e2e_logit_envelope, same_bits
from oracle.model import OracleDecoder
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth
from invariant_verify_gb300.verifier import DecoderVerifier, make_window, prefill_window

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


def _fresh_caches(cfg, n_slots, max_len):
    z = lambda: torch.zeros(n_slots, cfg.Hkv, max_len, cfg.hd, dtype=torch.bfloat16, device="cuda")
    return [(z(), z()) for _ in range(cfg.layers)]


@pytest.mark.parametrize("P", [1, 37, 300])
def test_prefill_equals_token_by_token(P):
    cfg = synth.DECODER2
    w = synth.decoder_weights_device(cfg)
    max_len = P + 8
    caches = _fresh_caches(cfg, 2, max_len)
    prompt = torch.randint(0, cfg.vocab, (P,), generator=synth.generator(60 + P), dtype=torch.int64).to(torch.int32)
    req = 4242
    pre = DecoderVerifier(cfg, w, caches, 2, max_len, P, P)
    pre.prefill(prefill_window(prompt, 0, req))
    torch.cuda.synchronize()
    one = DecoderVerifier(cfg, w, caches, 2, max_len, 1, 1)
    one.kc, one.vc = pre.kc, pre.vc                        # same cache tensors, slot 1
    targets = []
    for i in range(P):
        win = make_window(1, 1, prompt[i:i + 1], torch.tensor([i], dtype=torch.int32),
                          torch.tensor([req], dtype=torch.int32), prompt[i:i + 1])
        win.row_slot.fill_(1)
        one.prefill(win)
        targets.append(one.target.clone())
    torch.cuda.synchronize()
    for l in range(cfg.layers):
        assert same_bits(pre.kc[l][0, :, :P], pre.kc[l][1, :, :P]), f"layer {l} K"
        assert same_bits(pre.vc[l][0, :, :P], pre.vc[l][1, :, :P]), f"layer {l} V"
    assert torch.equal(pre.target.cpu(), torch.cat(targets).cpu())


def test_prefill_against_oracle():
    cfg = synth.DECODER2
    P = 128
    w = synth.decoder_weights_device(cfg)
    max_len = P + 8
    caches = _fresh_caches(cfg, 1, max_len)
    prompt = torch.randint(0, cfg.vocab, (P,), generator=synth.generator(61), dtype=torch.int64).to(torch.int32)
    win = prefill_window(prompt, 0, 77)
    ver = DecoderVerifier(cfg, w, caches, 1, max_len, P, P)
    ver.prefill(win)
    torch.cuda.synchronize()
    w_cpu = {k: v.cpu() for k, v in w.items()}
    orc = OracleDecoder(cfg, w_cpu, [(k.cpu() * 0, v.cpu() * 0) for k, v in caches], 1, max_len)
    slot, pos = np.zeros(P, np.int32), np.arange(P, dtype=np.int32)
    ref, tol = e2e_logit_envelope(orc, prompt.numpy(), slot, pos)
    agree = check_end_to_end(ver.logits.cpu().numpy(), ver.target.cpu().numpy(), ref, tol, win.row_req.cpu(), pos,
                             SEED, cfg.temperature, what="prefill")
    print(f"prefill: envelope {tol.min():.4f}..{tol.max():.4f}, token agreement {agree}/{P}")
    # the GPU's own logits give the GPU's tokens exactly
    assert np.array_equal(oracle.gumbel_argmax(ver.logits.cpu(), win.row_req.cpu(), win.row_pos.cpu(), SEED,
                                               cfg.temperature), ver.target.cpu().numpy())
