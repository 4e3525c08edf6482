"""The C-ABI library loads, exports every symbol include/biv.h declares, and
rejects bad arguments on the host before any CUDA call (no GPU needed).

Pointers used here are never dereferenced: every call below returns from
host-side validation before anything is enqueued.
"""
import ctypes as C
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "biv.h")

OK, NULL, SHAPE, ALIGN, VALUE, UNSUP = 0, 1, 2, 3, 4, 5
FAKE = 0x10000          # 16-byte aligned, never dereferenced
MISALIGNED = 0x10008


@pytest.fixture(scope="module")
def lib():
    from invariant_verify_gb300 import build, abi
    build.build()
    return abi.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(biv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(8):
        assert lib.biv_status_string(s)
    assert lib.biv_status_string(99) == b"unknown status"
    assert lib.biv_version() >= 100


def test_rmsnorm_validation(lib):
    f = lib.biv_rmsnorm
    assert f(None, None, None, 0, 1024, 1e-6, None) == OK
    assert f(None, None, None, 4, 1020, 1e-6, None) == SHAPE
    assert f(None, None, None, 4, 1024, -1.0, None) == VALUE
    assert f(None, None, None, 4, 1024, float("nan"), None) == VALUE
    assert f(None, None, None, 4, 1024, 1e-6, None) == NULL
    assert f(MISALIGNED, FAKE, FAKE, 4, 1024, 1e-6, None) == ALIGN
    a = lib.biv_add_rmsnorm
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1020, 1e-6, None) == SHAPE
    assert a(FAKE, None, FAKE, FAKE, FAKE, 4, 1024, 1e-6, None) == NULL
    assert a(FAKE, FAKE, FAKE, MISALIGNED, FAKE, 4, 1024, 1e-6, None) == ALIGN
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1024, 1e-6, None) == OK
    e = lib.biv_embed_rmsnorm
    assert e(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 0, 1e-6, None) == SHAPE
    assert e(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 10, 0.0, None) == VALUE


def test_gemm_validation(lib):
    f = lib.biv_gemm_nosplitk
    assert f(None, None, None, 0, 0, 64, 64, None) == OK
    assert f(None, None, None, 0, 4, 60, 64, None) == SHAPE
    assert f(None, None, None, 0, 4, 64, 60, None) == SHAPE
    assert f(None, None, None, 0, -1, 64, 64, None) == SHAPE
    assert f(None, None, None, 7, 4, 64, 64, None) == VALUE
    assert f(None, None, None, 0, 4, 64, 64, None) == NULL
    assert f(FAKE, MISALIGNED, FAKE, 1, 4, 64, 64, None) == ALIGN
    assert lib.biv_gemm_nosplitk_bn(FAKE, FAKE, FAKE, 0, 4, 64, 64, 40, None) == VALUE
    assert lib.biv_gemm_nosplitk_bn(FAKE, FAKE, FAKE, 0, 4, 64, 64, 272, None) == VALUE


def test_gemm_tile_width_rule(lib):
    for M in (1, 8, 64, 128):                       # one row tile: one wave of N tiles
        assert lib.biv_gemm_tile_n(M, 1024, 1024) == 16
        assert lib.biv_gemm_tile_n(M, 1536, 1024) == 16
        assert lib.biv_gemm_tile_n(M, 5632, 1024) == 48
        assert lib.biv_gemm_tile_n(M, 32000, 1024) == 224    # 143 tiles
        assert lib.biv_gemm_tile_n(M, 128256, 4096) == 224   # 573 tiles, 4 nearly full waves
    for M, N in ((1024, 4096), (256, 6144), (1024, 128256), (300, 1000)):
        bn = lib.biv_gemm_tile_n(M, N, 4096)
        assert 64 <= bn <= 256 and bn % 16 == 0
    assert lib.biv_gemm_tile_n(1024, 4096, 4096) == 224      # 8 x 19 = 152 tiles
    for M in (1, 1000):
        for N in (8, 24, 4096, 152064):
            bn = lib.biv_gemm_tile_n(M, N, 64)
            assert 16 <= bn <= 256 and bn % 16 == 0


def test_attention_validation_and_workspace(lib):
    ws = lib.biv_decode_attn_workspace_size
    # partials (hd floats) + max + sum per (row, head, split), + 16 B to align the partials to 32 B
    assert ws(64, 8, 2304) == 64 * 8 * 9 * 130 * 4 + 16
    assert ws(1, 1, 1) == 1 * 1 * 1 * 130 * 4 + 16
    assert ws(0, 8, 100) == 0
    f = lib.biv_decode_attn_fixedsplit
    args = lambda **kw: [kw.get(k, v) for k, v in [
        ("q", FAKE), ("kc", FAKE), ("vc", FAKE), ("slot", FAKE), ("pos", FAKE), ("o", FAKE), ("W", 16),
        ("rpg", 4), ("Hq", 8), ("Hkv", 2), ("hd", 128), ("n_slots", 4), ("max_len", 512), ("split", 256),
        ("ws", FAKE), ("ws_bytes", 1 << 30), ("stream", None)]]
    assert f(*args(hd=64)) == UNSUP
    assert f(*args(split=128)) == UNSUP
    assert f(*args(Hq=6, Hkv=4)) == SHAPE
    assert f(*args(ws_bytes=100)) == SHAPE
    assert f(*args(W=0)) == OK
    assert f(*args(q=None)) == NULL
    assert f(*args(o=MISALIGNED)) == ALIGN
    assert f(*args(rpg=0)) == SHAPE


def test_gqa_tile_rule(lib):
    golden = os.path.join(ROOT, "tests", "golden", "gqa_tile_rule.txt")
    rows = [list(map(int, l.split())) for l in open(golden) if l.strip() and not l.startswith("#")]
    for tile, G, D in rows:
        assert lib.biv_gqa_max_drafts(G, tile) == D
    assert lib.biv_gqa_max_drafts(0, 128) == -1
    assert lib.biv_gqa_max_drafts(256, 128) == -1
    assert lib.biv_gqa_max_drafts(4, 128) == 31


def test_kv_overwrite_validation(lib):
    f = lib.biv_kv_overwrite
    base = [FAKE, FAKE, FAKE, 256, FAKE, 1536, FAKE, FAKE, None, 16, 4, 2, 128, 4, 512, None]
    assert f(*base[:9], 0, *base[10:]) == OK
    b = list(base); b[9] = 15
    assert f(*b) == SHAPE                         # W % K != 0
    b = list(base); b[3] = 128
    assert f(*b) == SHAPE                         # k stride < Hkv*hd
    b = list(base); b[5] = 1540
    assert f(*b) == SHAPE                         # v stride not a multiple of 8
    b = list(base); b[2] = None
    assert f(*b) == NULL
    b = list(base); b[0] = MISALIGNED
    assert f(*b) == ALIGN


def test_select_and_accept_validation(lib):
    g = lib.biv_gumbel_argmax
    assert g(FAKE, 4, 30, 32, FAKE, FAKE, 1, 1.0, FAKE, None) == SHAPE      # V % 4
    assert g(FAKE, 4, 32, 30, FAKE, FAKE, 1, 1.0, FAKE, None) == SHAPE      # ld < V
    assert g(FAKE, 4, 32, 32, FAKE, FAKE, 1, -0.5, FAKE, None) == VALUE
    assert g(FAKE, 4, 32, 32, FAKE, FAKE, 1, math.inf, FAKE, None) == VALUE
    assert g(FAKE, 4, 32, 32, FAKE, FAKE, 1, math.nan, FAKE, None) == VALUE
    assert g(FAKE, 0, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, None) == OK
    assert g(None, 4, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, None) == NULL
    assert g(MISALIGNED, 4, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, None) == ALIGN
    big = (1 << 22) + 4                     # past the streaming kernel's block-maximum table
    assert g(FAKE, 4, big, big, FAKE, FAKE, 1, 1.0, FAKE, None) == UNSUP
    # the workspace entry: size = 64 B of counters + per heavy slot (R / 8 of them, at least one):
    # best key 8 B, row 4 B, units left 4 B (each 16-B aligned as arrays), units 16 B per
    # 8192-logit chunk, live blocks 2 B per 256-logit block
    wsz = lib.biv_gumbel_argmax_workspace_size
    al = lambda n: (n + 15) // 16 * 16
    for R, V in ((4096, 152064), (17, 1000), (3, 4)):
        cap, nb, nc = max(1, R // 8), -(-V // 256), -(-V // 8192)
        assert wsz(R, V) == 64 + al(cap * 8) + 2 * al(cap * 4) + cap * nc * 16 + al(cap * nb * 2)
    assert wsz(0, 32) == 0 and wsz(4, 30) == 0
    w = lib.biv_gumbel_argmax_ws
    ws = wsz(4, 32)
    assert w(FAKE, 4, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, None, ws, None) == NULL
    assert w(FAKE, 4, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, MISALIGNED, ws, None) == ALIGN
    assert w(FAKE, 4, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, FAKE, ws - 16, None) == SHAPE
    assert w(FAKE, 4, 30, 32, FAKE, FAKE, 1, 1.0, FAKE, FAKE, ws, None) == SHAPE
    assert w(FAKE, 0, 32, 32, FAKE, FAKE, 1, 1.0, FAKE, None, 0, None) == OK
    a = lib.biv_verify_accept
    assert a(FAKE, FAKE, FAKE, 4, 0, FAKE, FAKE, None) == SHAPE
    assert a(FAKE, FAKE, FAKE, 0, 4, FAKE, FAKE, None) == OK
    assert a(None, FAKE, FAKE, 4, 4, FAKE, FAKE, None) == NULL


def test_fused_entry_validation(lib):
    assert lib.biv_gemm_swiglu(FAKE, FAKE, FAKE, 4, 40, 64, None) == SHAPE        # F % 16
    assert lib.biv_gemm_swiglu(FAKE, FAKE, FAKE, 0, 48, 64, None) == OK
    assert lib.biv_gemm_swiglu(None, FAKE, FAKE, 4, 48, 64, None) == NULL
    assert lib.biv_swiglu_pack_weights(FAKE, FAKE, 48, 64, None) == VALUE         # in place
    assert lib.biv_swiglu_pack_weights(FAKE, FAKE + 4096, 40, 64, None) == SHAPE
    r = lib.biv_rope_kv_write
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 8, 4, 8, 2, 128, 4, 512, 10000.0, None]
    b = list(base); b[7] = 6
    assert r(*b) == SHAPE
    b = list(base); b[14] = 1.0
    assert r(*b) == VALUE
    b = list(base); b[1] = MISALIGNED
    assert r(*b) == ALIGN
    b = list(base); b[7] = 0
    assert r(*b) == OK


def test_lm_head_gumbel_validation(lib):
    f = lib.biv_lm_head_gumbel
    ws = lib.biv_lm_head_gumbel_workspace_size(64, 32000, 1024)
    assert ws == 64 * -(-32000 // lib.biv_gemm_tile_n(64, 32000, 1024)) * 8
    assert lib.biv_lm_head_gumbel_workspace_size(0, 32000, 1024) == 0
    base = [FAKE, FAKE, FAKE, 64, 32000, 1024, FAKE, FAKE, 1, 0.7, FAKE, FAKE, ws, None]
    b = list(base); b[4] = 32004
    assert f(*b) == SHAPE                       # N % 8
    b = list(base); b[9] = -1.0
    assert f(*b) == VALUE
    b = list(base); b[9] = math.nan
    assert f(*b) == VALUE
    b = list(base); b[12] = ws - 8
    assert f(*b) == SHAPE                       # workspace too small
    b = list(base); b[11] = None
    assert f(*b) == NULL
    b = list(base); b[2] = MISALIGNED
    assert f(*b) == ALIGN                       # logits, when given, aligned
    b = list(base); b[3] = 0
    assert f(*b) == OK


def test_lm_head_gumbel_accept_validation(lib):
    f = lib.biv_lm_head_gumbel_accept
    ws = lib.biv_lm_head_gumbel_workspace_size(64, 32000, 1024)
    #       A     B     logits M   N      K     req   pos   seed T    tok   draft p0    n  K  L     nl    ws    bytes s
    base = [FAKE, FAKE, FAKE, 64, 32000, 1024, FAKE, FAKE, 1, 0.7, FAKE, FAKE, FAKE, 8, 8, FAKE, FAKE, FAKE, ws, None]
    b = list(base); b[13] = 7
    assert f(*b) == SHAPE                       # M != n_req * rows_per_req
    b = list(base); b[14] = 0
    assert f(*b) == SHAPE
    b = list(base); b[4] = 32004
    assert f(*b) == SHAPE                       # N % 8
    b = list(base); b[9] = -1.0
    assert f(*b) == VALUE
    b = list(base); b[18] = ws - 8
    assert f(*b) == SHAPE                       # workspace too small
    for k in (11, 12, 15, 16, 17):
        b = list(base); b[k] = None
        assert f(*b) == NULL
    b = list(base); b[2] = MISALIGNED
    assert f(*b) == ALIGN
    b = list(base); b[3] = 0; b[13] = 0
    assert f(*b) == OK


def test_topk_and_ngram_validation(lib):
    t = lib.biv_gumbel_topk
    assert t(FAKE, 4, 32, 32, FAKE, FAKE, 1, 0.7, 0, FAKE, None) == SHAPE          # k < 1
    assert t(FAKE, 4, 32, 32, FAKE, FAKE, 1, 0.7, 65, FAKE, None) == SHAPE         # k > 64
    assert t(FAKE, 4, 8, 8, FAKE, FAKE, 1, 0.7, 9, FAKE, None) == SHAPE            # k > V
    assert t(FAKE, 4, 30, 32, FAKE, FAKE, 1, 0.7, 4, FAKE, None) == SHAPE          # V % 4
    assert t(FAKE, 4, 32, 32, FAKE, FAKE, 1, -1.0, 4, FAKE, None) == VALUE
    assert t(FAKE, 0, 32, 32, FAKE, FAKE, 1, 0.7, 4, FAKE, None) == OK
    assert t(MISALIGNED, 4, 32, 32, FAKE, FAKE, 1, 0.7, 4, FAKE, None) == ALIGN
    n = lib.biv_ngram_draft
    assert n(FAKE, 4, 100, FAKE, 3, 1, 0, FAKE, FAKE, None) == SHAPE               # K < 1
    assert n(FAKE, 4, 100, FAKE, 3, 1, 1025, FAKE, FAKE, None) == SHAPE
    assert n(FAKE, 4, 100, FAKE, 1, 2, 4, FAKE, FAKE, None) == VALUE               # n_max < n_min
    assert n(FAKE, 4, 100, FAKE, 65, 1, 4, FAKE, FAKE, None) == VALUE
    assert n(FAKE, 0, 100, FAKE, 3, 1, 4, FAKE, FAKE, None) == OK
    assert n(None, 4, 100, FAKE, 3, 1, 4, FAKE, FAKE, None) == NULL


def test_qkv_rope_validation(lib):
    f = lib.biv_gemm_qkv_rope
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, 64, 8, 1024, 8, 2, 128, 8, 4096, 10000.0, None]
    b = list(base); b[14] = 120
    assert f(*b) == SHAPE                       # hd % 16
    b = list(base); b[9] = 60
    assert f(*b) == SHAPE                       # W % K
    b = list(base); b[17] = 1.0
    assert f(*b) == VALUE
    b = list(base); b[5] = MISALIGNED
    assert f(*b) == ALIGN                       # qkv_out, when given
    b = list(base); b[2] = None
    assert f(*b) == NULL
    b = list(base); b[9] = 0
    assert f(*b) == OK
    p = lib.biv_rope_pack_qkv_weights
    assert p(FAKE, FAKE, 8, 2, 128, 1024, None) == VALUE          # in place
    assert p(FAKE, FAKE + 4096, 8, 2, 72, 1024, None) == SHAPE


def test_glue_validation(lib):
    assert lib.biv_embed(FAKE, FAKE, FAKE, 4, 100, 10, None) == SHAPE
    assert lib.biv_embed(FAKE, FAKE, FAKE, 0, 128, 10, None) == OK
    assert lib.biv_rope_qk(FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 127, 10000.0, None) == SHAPE
    assert lib.biv_rope_qk(FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 128, 0.5, None) == VALUE
    assert lib.biv_silu_mul(FAKE, FAKE, 4, 12, None) == SHAPE
    assert lib.biv_residual_add(FAKE, FAKE, FAKE, 12, None) == SHAPE
    assert lib.biv_residual_add(FAKE, FAKE, MISALIGNED, 16, None) == ALIGN


def test_noise_bucket_bounds_cover_the_oracle_noise(lib):
    # The selection kernel prunes with a host-side table of per-bucket noise
    # bounds; every one of the 2^23 noise values the oracle produces lies under
    # its bucket's bound (the GPU noise is checked bit-exact against these).
    import numpy as np
    import oracle
    from invariant_verify_gb300 import abi
    bounds = abi.biv_gumbel_bucket_bounds()
    words = np.arange(2 ** 23, dtype=np.uint32) << np.uint32(9)
    g = oracle.gumbel_from_words(words)
    assert np.all(g <= bounds[words >> 24])
    assert np.all(bounds - g.reshape(256, -1).max(axis=1) < 2e-3)
