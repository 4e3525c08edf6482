"""The no-alloc attention entry point against the workspace entry point.

Some callers cannot allocate device memory at all -- a host runtime that owns
every device allocation through its own pool, or a plugin that is handed
tensors but no allocator.  biv_decode_attn_fixedsplit_noalloc serves them: it
keeps the attention partials in a fixed scratch array inside the library
instead of a caller workspace.  This file checks, through the C ABI, that it
returns exactly the bits biv_decode_attn_fixedsplit returns on calls
enqueued back to back (so the scratch left by one call does not leak into
the next), and that a problem too large for the array is refused.

Kept in a file of its own that sorts last, so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from gpu_util import same_bits
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth

pytestmark = pytest.mark.gpu

BIV_ERR_SCRATCH = 8


def _case(n_slots, Hq, Hkv, p0, K, seed):
    g = synth.generator(seed)
    max_len = max(p0) + K + 30
    kc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g).cuda()
    vc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g).cuda()
    N = len(p0)
    q = synth.bf16_normal((N * K, Hq, 128), 1.0, g).cuda()
    slot = torch.as_tensor(np.repeat(np.arange(N), K), dtype=torch.int32).cuda()
    pos = torch.as_tensor(np.repeat(np.asarray(p0), K) + np.tile(np.arange(K), N), dtype=torch.int32).cuda()
    return q, kc, vc, slot, pos, K


def _with_workspace(q, kc, vc, slot, pos, rpg):
    W, Hq, _ = q.shape
    o = torch.full((W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.biv_decode_attn_workspace_size(W, Hq, kc.shape[2]), dtype=torch.uint8, device="cuda")
    B.biv_decode_attn_fixedsplit(q, kc, vc, slot, pos, o, rpg, ws)
    return o


def _no_alloc_into(o, q, kc, vc, slot, pos, rpg):
    B.biv_decode_attn_fixedsplit_noalloc(q, kc, vc, slot, pos, o, rpg)


def _nan_out(q):
    W, Hq, _ = q.shape
    return torch.full((W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")


def test_no_alloc_attention_matches_workspace_entry():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_verify_gb300 import build
    build.build()
    cases = [
        _case(4, 8, 2, [100, 255, 700, 1300], 8, seed=71),     # G=4, 8 rows per request
        _case(3, 8, 1, [900, 40, 1700], 8, seed=72),           # G=8, other positions and strides
    ]
    refs = [_with_workspace(*c) for c in cases]
    torch.cuda.synchronize()
    # The same kernels in the same order as the workspace entry point, so the
    # results are the same bits.  The two calls are enqueued back to back on
    # one stream with nothing in between (the second call's kernels may start
    # while the first call's last kernel finishes, on the same scratch), then
    # the first case again after the second overwrote the scratch.
    outs = [_nan_out(c[0]) for c in cases + cases[:1]]
    torch.cuda.synchronize()
    for o, c in zip(outs, cases + cases[:1]):
        _no_alloc_into(o, *c)
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs + refs[:1]):
        assert same_bits(o, ref)
    # a problem whose partials exceed the fixed scratch is refused, nothing launched
    big = B.biv_decode_attn_workspace_size(4096, 32, 8192)
    assert big > B.NOALLOC_SCRATCH_BYTES
    st = B.lib().biv_decode_attn_fixedsplit_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 4096,
                                                    16, 32, 8, 128, 64, 8192, 256, None)
    assert st == BIV_ERR_SCRATCH
    assert B.biv_device_error() == 0
