"""GPU parity of every libbiv kernel against the CPU oracle, and GPU-vs-GPU
batch invariance, through the C ABI.  Sizes span several tiles plus a
ragged tail; edge cases cover empty inputs and the degenerate shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, same_bits, dev
from invariant_verify_gb300 import abi as B
from invariant_verify_gb300 import synth

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


# ------------------------------------------------------------------ RMSNorm
@pytest.mark.parametrize("rows,d", [(1, 256), (16, 256), (64, 1024), (37, 4096), (5, 8), (3, 16384)])
def test_rmsnorm_parity(rows, d):
    g = synth.generator(rows * 7 + d)
    x = synth.bf16_normal((rows, d), 1.5, g)
    w = synth.bf16_normal((d,), 1.0, g)
    y = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    B.biv_rmsnorm(dev(x), dev(w), y, 1e-6)
    assert_close(y, oracle.rmsnorm(x, w, 1e-6), what="rmsnorm")


def test_rmsnorm_row_invariance_and_alias():
    x = dev(synth.bf16_normal((200, 1024), 1.0, synth.generator(3)))
    w = dev(torch.ones(1024, dtype=torch.bfloat16))
    full = torch.empty_like(x)
    B.biv_rmsnorm(x, w, full, 1e-6)
    for r in (0, 77, 199):
        one = torch.empty(1, 1024, dtype=torch.bfloat16, device="cuda")
        B.biv_rmsnorm(x[r:r + 1].contiguous(), w, one, 1e-6)
        assert same_bits(one[0], full[r])
    xa = x.clone()
    B.biv_rmsnorm(xa, w, xa, 1e-6)            # y may alias x
    assert same_bits(xa, full)
    B.biv_rmsnorm(x[:0], w, full[:0], 1e-6)   # empty


def test_fused_norms_equal_separate_kernels():
    g = synth.generator(17)
    for rows, d in ((64, 1024), (3, 4096), (16, 256)):
        x = dev(synth.bf16_normal((rows, d), 1.0, g))
        r = dev(synth.bf16_normal((rows, d), 0.3, g))
        w = dev(synth.bf16_normal((d,), 1.0, g))
        s_sum = torch.empty_like(x)
        s_norm = torch.empty_like(x)
        B.biv_residual_add(x, r, s_sum)
        B.biv_rmsnorm(s_sum, w, s_norm, 1e-6)
        f_sum = x.clone()
        f_norm = torch.empty_like(x)
        B.biv_add_rmsnorm(f_sum, r, w, f_sum, f_norm, 1e-6)      # x_out aliases x
        assert same_bits(f_sum, s_sum) and same_bits(f_norm, s_norm)
        table = dev(synth.bf16_normal((97, d), 1.0, g))
        tok = i32(np.arange(rows) * 7 % 97)
        e = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
        en = torch.empty_like(e)
        B.biv_embed(table, tok, e)
        B.biv_rmsnorm(e, w, en, 1e-6)
        fe = torch.empty_like(e)
        fen = torch.empty_like(e)
        B.biv_embed_rmsnorm(table, tok, w, fe, fen, 1e-6)
        assert same_bits(fe, e) and same_bits(fen, en)


# --------------------------------------------------------------------- GEMM
GEMM_SHAPES = [
    (1, 64, 64, torch.bfloat16, None),
    (3, 136, 72, torch.bfloat16, None),        # ragged N (not a tile multiple), K < one k-block
    (130, 520, 200, torch.bfloat16, None),     # two row tiles + ragged M, ragged K
    (64, 1536, 1024, torch.bfloat16, None),
    (16, 2048, 256, torch.float32, None),
    (300, 1000, 520, torch.float32, None),
    (257, 384, 128, torch.bfloat16, 256),
    (129, 200, 136, torch.float32, 128),
    (77, 96, 64, torch.bfloat16, 32),
    (45, 48, 64, torch.float32, 16),
    (200, 640, 192, torch.bfloat16, 64),
]


@pytest.mark.parametrize("M,N,K,dt,bn", GEMM_SHAPES)
def test_gemm_parity(M, N, K, dt, bn):
    g = synth.generator(M * 131 + N * 7 + K)
    A = synth.bf16_normal((M, K), 1.0, g)
    Bw = synth.bf16_normal((N, K), 0.05, g)
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    B.biv_gemm_nosplitk(dev(A), dev(Bw), C, bn=bn)
    assert_close(C, oracle.gemm(A, Bw), what=f"gemm {M}x{N}x{K}")


def test_gemm_empty_and_single():
    A = dev(synth.bf16_normal((0, 64), 1.0, synth.generator(1)))
    Bw = dev(synth.bf16_normal((64, 64), 1.0, synth.generator(2)))
    C = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm_nosplitk(A, Bw, C)


def test_gemm_rows_are_batch_invariant():
    g = synth.generator(11)
    A = dev(synth.bf16_normal((300, 1024), 1.0, g))
    Bw = dev(synth.bf16_normal((1536, 1024), 0.05, g))
    full = torch.empty(300, 1536, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(A, Bw, full)
    for M in (1, 2, 7, 64, 128, 129, 256):
        part = torch.empty(M, 1536, dtype=torch.float32, device="cuda")
        B.biv_gemm_nosplitk(A[:M].contiguous(), Bw, part)
        assert same_bits(part, full[:M]), M
    perm = torch.randperm(300, generator=synth.generator(5)).cuda()
    pc = torch.empty_like(full)
    B.biv_gemm_nosplitk(A[perm].contiguous(), Bw, pc)
    assert same_bits(pc, full[perm])
    # a row placed at every slot of a 128-row tile gives the same bits
    row = A[5:6].repeat(128, 1).contiguous()
    rc = torch.empty(128, 1536, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(row, Bw, rc)
    assert same_bits(rc, full[5:6].repeat(128, 1))


def test_gemm_tile_width_does_not_change_bits():
    g = synth.generator(12)
    A = dev(synth.bf16_normal((150, 2048), 1.0, g))
    Bw = dev(synth.bf16_normal((512, 2048), 0.05, g))
    outs = {}
    for bn in (16, 32, 64, 128, 256):
        C = torch.empty(150, 512, dtype=torch.float32, device="cuda")
        B.biv_gemm_nosplitk(A, Bw, C, bn=bn)
        outs[bn] = C
    for bn in (16, 32, 64, 128):
        assert same_bits(outs[bn], outs[256]), bn


@pytest.mark.parametrize("M,F,K", [(64, 2816, 1024), (1, 48, 64), (130, 1024, 200), (300, 112, 136),
                                   (300, 1040, 256)])            # the last: 256-row CTA-pair tiles
def test_gemm_swiglu_equals_gemm_then_silu(M, F, K):
    g = synth.generator(M + F + K)
    A = dev(synth.bf16_normal((M, K), 1.0, g))
    wgu = dev(synth.bf16_normal((2 * F, K), 0.05, g))
    gu = torch.empty(M, 2 * F, dtype=torch.bfloat16, device="cuda")
    ref = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    B.biv_gemm_nosplitk(A, wgu, gu)
    B.biv_silu_mul(gu, ref)
    packed = torch.empty_like(wgu)
    B.biv_swiglu_pack_weights(wgu, packed)
    act = torch.full((M, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.biv_gemm_swiglu(A, packed, act)
    assert same_bits(act, ref)


# --------------------------------------------------------------- attention
def _attn_case(n_slots, Hq, Hkv, max_len, p0, K, seed):
    g = synth.generator(seed)
    kc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g)
    vc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g)
    N = len(p0)
    W = N * K
    q = synth.bf16_normal((W, Hq, 128), 1.0, g)
    slot = np.repeat(np.arange(N), K)
    pos = np.repeat(np.asarray(p0), K) + np.tile(np.arange(K), N)
    return q, kc, vc, slot.astype(np.int32), pos.astype(np.int32)


def _run_attn(q, kc, vc, slot, pos, rpg):
    W, Hq, _ = q.shape
    o = torch.full((W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.biv_decode_attn_workspace_size(W, Hq, kc.shape[2]), dtype=torch.uint8, device="cuda")
    B.biv_decode_attn_fixedsplit(q, kc, vc, i32(slot), i32(pos), o, rpg, ws)
    return o


@pytest.mark.parametrize("Hq,Hkv,K,p0", [
    (8, 2, 8, [250, 511, 1000]),        # G=4, windows straddling the 256 / 512 split edges
    (32, 1, 4, [0, 300, 767]),          # G=32: 4 rows x 32 heads = one full 128-row tile
    (8, 1, 16, [100, 1030]),            # G=8: 16 x 8 = 128
    (8, 1, 20, [5, 600]),               # G=8, K=20: two tiles per request
    (4, 4, 3, [255, 256, 257]),         # G=1
])
def test_attention_parity(Hq, Hkv, K, p0):
    max_len = max(p0) + K + 40
    q, kc, vc, slot, pos = _attn_case(len(p0), Hq, Hkv, max_len, p0, K, seed=Hq * 100 + K)
    o = _run_attn(dev(q), dev(kc), dev(vc), slot, pos, K)
    ref = oracle.attention(q, kc, vc, slot, pos)
    assert_close(o, ref, what="attention")


def test_attention_rows_are_batch_invariant():
    q, kc, vc, slot, pos = _attn_case(4, 8, 2, 1400, [100, 255, 700, 1300], 8, seed=9)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    full = _run_attn(qd, kd, vd, slot, pos, 8)
    alone = _run_attn(qd, kd, vd, slot, pos, 1)          # every row in its own tile
    assert same_bits(alone, full)
    for w in (0, 9, 31):                                  # a single-row call
        one = _run_attn(qd[w:w + 1].contiguous(), kd, vd, slot[w:w + 1], pos[w:w + 1], 1)
        assert same_bits(one[0], full[w])
    perm = np.random.default_rng(1).permutation(32)
    pq = _run_attn(qd[torch.as_tensor(perm).cuda()].contiguous(), kd, vd, slot[perm], pos[perm], 1)
    assert same_bits(pq, full[torch.as_tensor(perm).cuda()])
    # stale values after a row's position do not change it
    kd2, vd2 = kd.clone(), vd.clone()
    for r, p in enumerate([100, 255, 700, 1300]):
        kd2[r, :, p + 8:] = 7.0
        vd2[r, :, p + 8:] = -3.0
    assert same_bits(_run_attn(qd, kd2, vd2, slot, pos, 8), full)
    # ... not even NaN (keys past the last one any row reads are never multiplied in)
    kd3, vd3 = kd.clone(), vd.clone()
    for r, p in enumerate([100, 255, 700, 1300]):
        kd3[r, :, p + 8:] = float("nan")
        vd3[r, :, p + 8:] = float("nan")
    assert same_bits(_run_attn(qd, kd3, vd3, slot, pos, 8), full)


def test_attention_rows_invariant_across_mma_shapes():
    """A full 128-row tile (G = 8 heads x 16 rows: 128-row MMAs) and the same
    rows one at a time (8 rows: 64-row MMAs) give the same bits, splits with a
    ragged last 16-key step included."""
    q, kc, vc, slot, pos = _attn_case(3, 8, 1, 1100, [5, 290, 1000], 16, seed=19)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    full = _run_attn(qd, kd, vd, slot, pos, 16)
    alone = _run_attn(qd, kd, vd, slot, pos, 1)
    assert same_bits(alone, full)


def test_attention_past_the_tile_tables_same_bits():
    """Past 2048 row tiles the split kernel numbers all (split, KV head, tile)
    triples and skips the dead ones instead of dealing out live items from
    its shared-memory tables; rows read their positions from global memory.
    The same rows give the same bits either way, and match the oracle."""
    W, Hq, Hkv, max_len = 2050, 2, 2, 300
    g = synth.generator(2050)
    kc = synth.bf16_normal((4, Hkv, max_len, 128), 1.0, g)
    vc = synth.bf16_normal((4, Hkv, max_len, 128), 1.0, g)
    q = synth.bf16_normal((W, Hq, 128), 1.0, g)
    slot = (np.arange(W) % 4).astype(np.int32)
    pos = (np.arange(W) * 37 % 290).astype(np.int32)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    many = _run_attn(qd, kd, vd, slot, pos, 1)            # 2050 tiles: dense numbering
    few = _run_attn(qd[:2048].contiguous(), kd, vd, slot[:2048], pos[:2048], 1)
    assert same_bits(many[:2048], few)
    rows = [0, 1000, 2049]
    ref = oracle.attention(q[rows], kc, vc, slot[rows], pos[rows])
    assert_close(many[rows], ref, what="attention (dense numbering)")


def test_attention_two_item_and_one_item_kernels_same_bits():
    """Windows whose tile tables fit beside two warpgroups' buffers run two
    items per SM (attn_pp_kernel); 2000 one-row tiles do not, and run one
    item per SM (attn_tc_kernel, tables still in shared memory).  The same
    rows give the same bits either way, and match the oracle."""
    W, Hq, Hkv, max_len = 2000, 8, 2, 1200
    g = synth.generator(2000)
    kc = synth.bf16_normal((8, Hkv, max_len, 128), 1.0, g)
    vc = synth.bf16_normal((8, Hkv, max_len, 128), 1.0, g)
    q = synth.bf16_normal((W, Hq, 128), 1.0, g)
    slot = (np.arange(W) % 8).astype(np.int32)
    pos = (np.arange(W) * 131 % 1150).astype(np.int32)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    big = _run_attn(qd, kd, vd, slot, pos, 1)             # one item per SM
    small = _run_attn(qd[:256].contiguous(), kd, vd, slot[:256], pos[:256], 1)   # two per SM
    assert same_bits(big[:256], small)
    rows = [0, 77, 255, 1999]
    ref = oracle.attention(q[rows], kc, vc, slot[rows], pos[rows])
    assert_close(big[rows], ref, what="attention (one item per SM)")


@pytest.mark.parametrize("W", [4096, 4352])
def test_attention_combine_many_pairs_per_warp(W):
    """W x 32 heads (row, head) pairs, many per combine warp.  At W = 4096 the
    combine deals the pairs by cost (the largest window with that deal); at
    W = 4352 it deals them round-robin and a warp reads the slots and
    positions of its pairs in several rounds of 32.  Sampled rows match the
    oracle, and the first 1024 rows give the same bits when they are the whole
    window (about nine pairs per combine warp: the balanced deal)."""
    Hq, Hkv, K, n_slots, max_len = 32, 8, 16, 16, 700
    g = synth.generator(4096)
    kc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g)
    vc = synth.bf16_normal((n_slots, Hkv, max_len, 128), 1.0, g)
    q = synth.bf16_normal((W, Hq, 128), 1.0, g)
    req = np.arange(W) // K
    slot = (req % n_slots).astype(np.int32)
    pos = ((req * 37) % 600 + 40 + np.arange(W) % K).astype(np.int32)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    big = _run_attn(qd, kd, vd, slot, pos, K)
    small = _run_attn(qd[:1024].contiguous(), kd, vd, slot[:1024], pos[:1024], K)
    assert same_bits(big[:1024], small)
    rows = [0, 15, 2047, 3000, W - 1]
    ref = oracle.attention(q[rows], kc, vc, slot[rows], pos[rows])
    assert_close(big[rows], ref, what=f"attention, {W * Hq} pairs")
    assert not torch.isnan(big.float()).any()


def test_attention_bad_position_raises_device_error():
    q, kc, vc, slot, pos = _attn_case(2, 8, 2, 600, [100, 300], 4, seed=12)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    good = _run_attn(qd, kd, vd, slot, pos, 4)
    assert B.biv_device_error() == 0
    bad = pos.copy()
    bad[5] = 600                                           # one past the cache
    o = _run_attn(qd, kd, vd, slot, bad, 4)
    assert B.biv_device_error() & 2                        # BIV_DEVERR_INDEX, and the flag is cleared
    assert torch.count_nonzero(o[5]) == 0                  # the bad row is zeroed
    keep = [w for w in range(8) if w != 5]
    assert same_bits(o[keep], good[keep])                  # the other rows are unaffected


def test_attention_bad_rows_with_the_balanced_combine():
    """64 requests x 16 rows x 32 heads: enough (row, head) pairs per combine
    warp for the cost deal.  Rows with a position past the cache are zeroed
    (costing one unit each in the deal) and raise the device flag; every other
    row keeps the bits of the clean window."""
    p0 = [(37 * r) % 500 + 20 for r in range(64)]
    q, kc, vc, slot, pos = _attn_case(64, 32, 8, 560, p0, 16, seed=31)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    good = _run_attn(qd, kd, vd, slot, pos, 16)
    assert B.biv_device_error() == 0
    bad = pos.copy()
    rows = [3, 400, 401, 1023]
    bad[rows] = 560                                        # one past the cache
    o = _run_attn(qd, kd, vd, slot, bad, 16)
    assert B.biv_device_error() & 2                        # BIV_DEVERR_INDEX, and the flag is cleared
    assert torch.count_nonzero(o[rows]) == 0
    keep = [w for w in range(1024) if w not in rows]
    assert same_bits(o[keep], good[keep])
    ref = oracle.attention(q[[0, 700]], kc, vc, slot[[0, 700]], pos[[0, 700]])
    assert_close(good[[0, 700]], ref, what="attention, balanced combine")


@pytest.mark.parametrize("n_req,K,Hq,Hkv", [(2, 4, 8, 2), (64, 16, 32, 8)])   # round-robin / balanced combine
def test_attention_row_outside_its_slot_group(n_req, K, Hq, Hkv):
    """A row whose slot differs from its group's first row (rows of one group
    must share a cache slot) raises BIV_DEVERR_GROUP and is zeroed; the other
    rows of its group and of the window keep the bits of the clean window."""
    p0 = [(53 * r) % 400 + 30 for r in range(n_req)]
    q, kc, vc, slot, pos = _attn_case(n_req, Hq, Hkv, 480, p0, K, seed=17 + n_req)
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    good = _run_attn(qd, kd, vd, slot, pos, K)
    assert B.biv_device_error() == 0
    bad = slot.copy()
    w = 2                                                  # not the first row of group 0
    bad[w] = 1                                             # another request's slot
    o = _run_attn(qd, kd, vd, bad, pos, K)
    assert B.biv_device_error() & 4                        # BIV_DEVERR_GROUP, and the flag is cleared
    assert torch.count_nonzero(o[w]) == 0
    keep = [r for r in range(n_req * K) if r != w]
    assert same_bits(o[keep], good[keep])


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """Failure detection without a fault: a kernel waits, through the
    library's bounded wait, on a barrier nothing completes; it gives up,
    raises BIV_DEVERR_TIMEOUT and returns.  Kernels launched afterwards run
    and match the oracle."""
    assert B.biv_device_error() == 0
    B.biv_selftest_wait_timeout()
    assert B.biv_device_error() & 1                        # BIV_DEVERR_TIMEOUT, and the flag is cleared
    assert B.biv_device_error() == 0
    g = synth.generator(99)
    A = synth.bf16_normal((37, 256), 1.0, g)
    Bw = synth.bf16_normal((192, 256), 0.1, g)
    C_ = torch.empty(37, 192, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(dev(A), dev(Bw), C_)
    assert_close(C_, oracle.gemm(A, Bw), what="GEMM after a timed-out wait")
    assert B.biv_device_error() == 0


def test_attention_first_position():
    q, kc, vc, slot, pos = _attn_case(2, 4, 2, 64, [0, 0], 1, seed=4)
    o = _run_attn(dev(q), dev(kc), dev(vc), slot, pos, 1)
    v = oracle.from_bf16(vc)
    for w in range(2):
        for h in range(4):
            assert_close(o[w, h], v[w, h // 2, 0], tol=1e-2)


# -------------------------------------------------------------- KV + glue
def test_kv_overwrite_bit_exact_and_rows_keep():
    g = synth.generator(21)
    kc = synth.bf16_normal((3, 2, 64, 128), 1.0, g)
    vc = synth.bf16_normal((3, 2, 64, 128), 1.0, g)
    kn = synth.bf16_normal((12, 2 * 128), 1.0, g)
    vbig = synth.bf16_normal((12, 1536), 1.0, g)                 # strided source
    vn = vbig[:, 1280:]
    slot = np.repeat([2, 0, 1], 4).astype(np.int32)
    pos = (np.repeat([10, 50, 0], 4) + np.tile(np.arange(4), 3)).astype(np.int32)
    kd, vd = dev(kc), dev(vc)
    B.biv_kv_overwrite(kd, vd, dev(kn), dev(vbig)[:, 1280:], i32(slot), i32(pos), K=4)
    ko = oracle._np(kc).copy(); vo = oracle._np(vc).copy()
    oracle.kv_overwrite(ko, vo, oracle._np(kn).reshape(12, 2, 128), oracle._np(vn.contiguous()).reshape(12, 2, 128),
                        slot, pos)
    assert np.array_equal(oracle._np(kd.cpu()), ko) and np.array_equal(oracle._np(vd.cpu()), vo)
    # rows_keep: request r writes only its first keep[r] rows
    kd, vd = dev(kc), dev(vc)
    keep = np.array([1, 4, 0], np.int32)
    B.biv_kv_overwrite(kd, vd, dev(kn), dev(vbig)[:, 1280:], i32(slot), i32(pos), K=4, rows_keep=i32(keep))
    rows = [w for w in range(12) if w % 4 < keep[w // 4]]
    ko = oracle._np(kc).copy(); vo = oracle._np(vc).copy()
    oracle.kv_overwrite(ko, vo, oracle._np(kn).reshape(12, 2, 128)[rows],
                        oracle._np(vn.contiguous()).reshape(12, 2, 128)[rows], slot[rows], pos[rows])
    assert np.array_equal(oracle._np(kd.cpu()), ko) and np.array_equal(oracle._np(vd.cpu()), vo)


def test_rope_kv_write_equals_rope_then_overwrite():
    W, K, Hq, Hkv, hd = 12, 4, 8, 2, 128
    g = synth.generator(61)
    qkv = dev(synth.bf16_normal((W, (Hq + 2 * Hkv) * hd), 1.0, g))
    kc = dev(synth.bf16_normal((3, Hkv, 80, hd), 1.0, g))
    vc = dev(synth.bf16_normal((3, Hkv, 80, hd), 1.0, g))
    slot = i32(np.repeat([2, 0, 1], K))
    pos = i32(np.repeat([10, 50, 0], K) + np.tile(np.arange(K), 3))
    for keep in (None, i32([1, 4, 0])):
        q1 = torch.empty(W, Hq, hd, dtype=torch.bfloat16, device="cuda")
        k1 = torch.empty(W, Hkv * hd, dtype=torch.bfloat16, device="cuda")
        kc1, vc1 = kc.clone(), vc.clone()
        B.biv_rope_qk(qkv, q1, k1, pos, Hq, Hkv, hd, 10000.0)
        B.biv_kv_overwrite(kc1, vc1, k1, qkv[:, (Hq + Hkv) * hd:], slot, pos, K=K, rows_keep=keep)
        q2 = torch.empty_like(q1)
        kc2, vc2 = kc.clone(), vc.clone()
        B.biv_rope_kv_write(qkv, q2, kc2, vc2, slot, pos, Hq, 10000.0, K=K, rows_keep=keep)
        assert same_bits(q2, q1) and same_bits(kc2, kc1) and same_bits(vc2, vc1)


@pytest.mark.parametrize("W,K,d,Hq,Hkv,hd", [(12, 4, 256, 8, 2, 128), (64, 8, 1024, 8, 2, 128),
                                             (130, 1, 512, 4, 4, 64), (256, 256, 4096, 32, 8, 128),
                                             (40, 8, 512, 4, 2, 256),          # 16 frequency groups
                                             (1024, 16, 4096, 32, 8, 128)])    # the bench's window: CTA pairs, two waves
def test_qkv_rope_gemm_equals_gemm_then_rope_kv_write(W, K, d, Hq, Hkv, hd):
    g = synth.generator(W + d)
    n_slots, max_len = W // K + 1, 400
    A = dev(synth.bf16_normal((W, d), 1.0, g))
    wqkv = dev(synth.bf16_normal(((Hq + 2 * Hkv) * hd, d), 0.02, g))
    kc = dev(synth.bf16_normal((n_slots, Hkv, max_len, hd), 1.0, g))
    vc = dev(synth.bf16_normal((n_slots, Hkv, max_len, hd), 1.0, g))
    groups = W // K
    slot = i32(np.repeat(np.arange(groups)[::-1], K))
    base = np.random.default_rng(W).integers(0, max_len - K, groups)
    pos = i32(np.repeat(base, K) + np.tile(np.arange(K), groups))
    packed = torch.empty_like(wqkv)
    B.biv_rope_pack_qkv_weights(wqkv, packed, Hq, Hkv, hd)
    keeps = [None] + ([i32(np.random.default_rng(1).integers(0, K + 1, groups))] if K > 1 else [])
    for keep in keeps:
        for theta in (10000.0, 500000.0):
            qkv = torch.empty(W, (Hq + 2 * Hkv) * hd, dtype=torch.bfloat16, device="cuda")
            B.biv_gemm_nosplitk(A, wqkv, qkv)
            q1 = torch.empty(W, Hq, hd, dtype=torch.bfloat16, device="cuda")
            kc1, vc1 = kc.clone(), vc.clone()
            B.biv_rope_kv_write(qkv, q1, kc1, vc1, slot, pos, Hq, theta, K=K, rows_keep=keep)
            q2 = torch.empty_like(q1)
            kc2, vc2 = kc.clone(), vc.clone()
            qkv2 = torch.empty_like(qkv)
            B.biv_gemm_qkv_rope(A, packed, q2, kc2, vc2, slot, pos, theta, K=K, rows_keep=keep, qkv_out=qkv2)
            assert same_bits(qkv2, qkv)
            assert same_bits(q2, q1) and same_bits(kc2, kc1) and same_bits(vc2, vc1)
            # without the projection copy
            q3 = torch.empty_like(q1)
            kc3, vc3 = kc.clone(), vc.clone()
            B.biv_gemm_qkv_rope(A, packed, q3, kc3, vc3, slot, pos, theta, K=K, rows_keep=keep)
            assert same_bits(q3, q1) and same_bits(kc3, kc1) and same_bits(vc3, vc1)


def test_rope_parity():
    W, Hq, Hkv, hd = 10, 8, 2, 128
    g = synth.generator(31)
    qkv = synth.bf16_normal((W, (Hq + 2 * Hkv) * hd), 1.0, g)
    pos = np.array([0, 1, 7, 100, 255, 256, 1000, 2047, 4095, 8191], np.int32)
    q = torch.empty(W, Hq, hd, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(W, Hkv * hd, dtype=torch.bfloat16, device="cuda")
    for theta in (10000.0, 500000.0):
        B.biv_rope_qk(dev(qkv), q, k, i32(pos), Hq, Hkv, hd, theta)
        x = oracle.from_bf16(qkv)
        assert_close(q, oracle.rope(x[:, :Hq * hd].reshape(W, Hq, hd), pos, theta), what="rope q")
        assert_close(k.view(W, Hkv, hd), oracle.rope(x[:, Hq * hd:(Hq + Hkv) * hd].reshape(W, Hkv, hd), pos, theta),
                     what="rope k")


def test_silu_mul_residual_embed_parity():
    g = synth.generator(41)
    gu = synth.bf16_normal((33, 2 * 2816), 2.0, g)
    out = torch.empty(33, 2816, dtype=torch.bfloat16, device="cuda")
    B.biv_silu_mul(dev(gu), out)
    assert_close(out, oracle.silu_mul(gu), what="silu")
    x = synth.bf16_normal((33, 1024), 1.0, g)
    y = synth.bf16_normal((33, 1024), 1.0, g)
    o = torch.empty(33, 1024, dtype=torch.bfloat16, device="cuda")
    B.biv_residual_add(dev(x), dev(y), o)
    assert_close(o, oracle.from_bf16(x) + oracle.from_bf16(y), tol=4e-3, what="residual")
    table = synth.bf16_normal((500, 1024), 1.0, g)
    tok = np.array([0, 499, 17, 17, 250], np.int32)
    e = torch.empty(5, 1024, dtype=torch.bfloat16, device="cuda")
    B.biv_embed(dev(table), i32(tok), e)
    assert torch.equal(e.cpu(), table[tok])


# -------------------------------------------------------------- selection
def test_noise_bit_exact_over_every_uniform():
    words = np.arange(2 ** 23, dtype=np.uint32) << np.uint32(9)
    g = torch.empty(2 ** 23, dtype=torch.float32, device="cuda")
    B.biv_gumbel_from_words(torch.from_numpy(words.view(np.int32)).cuda(), g)
    ref = oracle.gumbel_from_words(words)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # random full 32-bit words, low bits included
    w = torch.randint(-2 ** 31, 2 ** 31 - 1, (1 << 20,), generator=synth.generator(5), dtype=torch.int64)
    w = w.to(torch.int32)
    g = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
    B.biv_gumbel_from_words(w.cuda(), g)
    ref = oracle.gumbel_from_words(w.numpy().view(np.uint32))
    assert np.array_equal(g.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_noise_bucket_bounds_hold_for_every_word():
    # The selection kernel's pruning bound: noise(word) <= bounds[word >> 24]
    # for all 2^23 uniforms (the low 9 bits do not change the uniform).
    words = np.arange(2 ** 23, dtype=np.uint32) << np.uint32(9)
    g = torch.empty(2 ** 23, dtype=torch.float32, device="cuda")
    B.biv_gumbel_from_words(torch.from_numpy(words.view(np.int32)).cuda(), g)
    bounds = B.biv_gumbel_bucket_bounds()
    gb = g.cpu().numpy()
    assert np.all(gb <= bounds[words >> 24])
    # and the bound is tight enough to prune: within 2e-3 of each bucket's top
    top = gb.reshape(256, -1).max(axis=1)
    assert np.all(bounds - top < 2e-3)


def test_noise_rows_bit_exact():
    req = np.array([0, 7, 2 ** 31 - 1, 123456], np.int64)
    pos = np.array([0, 99, 4095, 131071], np.int32)
    V = 5000
    g = torch.empty(4, V, dtype=torch.float32, device="cuda")
    B.biv_gumbel_noise(SEED, i32(req), i32(pos), g)
    for r in range(4):
        ref = oracle.gumbel_row(SEED, int(req[r]), int(pos[r]) + 1, V)
        assert np.array_equal(g[r].cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("R,V,T,std", [
    (16, 2048, 1.0, 1.0), (64, 32000, 0.7, 0.64), (37, 152064, 0.7, 3.0), (5, 4, 1.0, 1.0),
    (9, 12, 0.5, 1.0), (33, 2052, 2.0, 5.0), (8, 32000, 0.0, 1.0), (3, 100, 1e-3, 1.0)])
def test_gumbel_argmax_bit_exact(R, V, T, std):
    g = synth.generator(R * 1000 + V)
    x = torch.randn(R, V, generator=g) * std
    req = torch.randint(0, 2 ** 31 - 1, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    pos = torch.randint(0, 8000, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    tok = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(x.cuda(), req.cuda(), pos.cuda(), SEED, T, tok)
    ref = oracle.gumbel_argmax(x, req, pos, SEED, T)
    assert np.array_equal(tok.cpu().numpy(), ref)


def test_gumbel_argmax_peaked_ties_and_stride():
    cfg = synth.SELECT
    x, kind = synth.select_logits(cfg, rows=48, seed=3)
    xt, _ = synth.select_logits(cfg, rows=48, seed=3, exact_ties=True)
    req = torch.arange(48, dtype=torch.int32)
    pos = torch.arange(48, dtype=torch.int32) * 3
    for logits, T in ((x, 0.7), (x, 0.0), (xt, 0.0), (xt, 0.7)):
        tok = torch.empty(48, dtype=torch.int32, device="cuda")
        B.biv_gumbel_argmax(logits.cuda(), req.cuda(), pos.cuda(), SEED, T, tok)
        assert np.array_equal(tok.cpu().numpy(), oracle.gumbel_argmax(logits, req, pos, SEED, T))
    # a leading dimension larger than V: only the first V columns count
    pad = torch.full((48, cfg.vocab + 4), 1e30)
    pad[:, :cfg.vocab] = x
    tok = torch.empty(48, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(pad.cuda(), req.cuda(), pos.cuda(), SEED, 0.7, tok, V=cfg.vocab)
    assert np.array_equal(tok.cpu().numpy(), oracle.gumbel_argmax(x, req, pos, SEED, 0.7))
    B.biv_gumbel_argmax(pad[:0].cuda(), req[:0].cuda(), pos[:0].cuda(), SEED, 0.7, tok[:0], V=cfg.vocab)


def _many_rows():
    """A row count that sends the selection to its streaming kernel (two or
    more rows per SM); fewer rows go to the eight-CTA cluster kernel."""
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count + 5


@pytest.mark.parametrize("V,T", [(8196, 0.7), (4, 1.0), (24580, 0.0), (16388, 2.0), (1000, 1e-3)])
def test_gumbel_argmax_streaming_rows_bit_exact(V, T):
    """Many rows: one CTA per row, ring of bulk copies, block maxima, pass 2
    over live blocks.  V spans several 8192-logit chunks and a ragged tail;
    rows mix flat, peaked, NaN-holding, all-NaN, -inf and exact-tie rows."""
    R = _many_rows()
    g = synth.generator(V + 11)
    x = torch.randn(R, V, generator=g) * 2.0
    x[1::5, V // 3] += 40.0                       # peaked rows
    x[2::7, :] = float("nan")                     # all-NaN rows select token 0
    x[3::7, ::3] = float("nan")                   # scattered NaN never wins
    x[4::9, :] = float("-inf")
    x[4::9, V - 1] = 0.0                          # a single finite logit at the tail
    x[5::11, :] = 1.5                             # exact ties everywhere
    req = torch.randint(0, 2 ** 31 - 1, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    pos = torch.randint(0, 8000, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    tok = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(x.cuda(), req.cuda(), pos.cuda(), SEED, T, tok)
    assert np.array_equal(tok.cpu().numpy(), oracle.gumbel_argmax(x, req, pos, SEED, T))
    # the same rows through the cluster kernel (few rows) and with a padded
    # leading dimension: identical tokens
    sub = [0, 1, 2, 3, 4, 5, R - 1]
    few = torch.empty(len(sub), dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(x[sub].cuda(), req[sub].cuda(), pos[sub].cuda(), SEED, T, few)
    assert torch.equal(few, tok[sub])
    pad = torch.full((R, V + 12), 1e30)
    pad[:, :V] = x
    tp = torch.empty(R, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(pad.cuda(), req.cuda(), pos.cuda(), SEED, T, tp, V=V)
    assert torch.equal(tp, tok)
    # with a workspace (flat rows handed to the unit kernel): the same tokens,
    # also with a padded leading dimension and a workspace full of stale bytes
    ws = torch.full((B.biv_gumbel_argmax_workspace_size(R, V),), 0xA5, dtype=torch.uint8, device="cuda")
    tw = torch.full((R,), -3, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax_ws(x.cuda(), req.cuda(), pos.cuda(), SEED, T, tw, ws)
    assert torch.equal(tw, tok)
    tw.fill_(-3)
    B.biv_gumbel_argmax_ws(pad.cuda(), req.cuda(), pos.cuda(), SEED, T, tw, ws, V=V)
    assert torch.equal(tw, tok)


def test_gumbel_argmax_streaming_rows_concurrent_streams_and_graph_replays():
    """The streaming kernel deals rows out by a per-launch ticket counter that
    the launch's last CTA resets: back-to-back launches, launches on two
    streams at once and graph replays all select every row exactly."""
    R, V = _many_rows() + 40, 16384
    g = synth.generator(321)
    xs = [torch.randn(R, V, generator=g) * 3.0 for _ in range(2)]
    req = torch.randint(0, 2 ** 31 - 1, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    pos = torch.randint(0, 8000, (R,), generator=g, dtype=torch.int64).to(torch.int32)
    refs = [oracle.gumbel_argmax(x, req, pos, SEED, 0.7) for x in xs]
    xd = [x.cuda() for x in xs]
    rq, ps = req.cuda(), pos.cuda()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    toks = [torch.full((R,), -7, dtype=torch.int32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(5):
        for i in range(2):
            toks[i].fill_(-7)
        torch.cuda.synchronize()
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                for _ in range(3):
                    B.biv_gumbel_argmax(xd[i], rq, ps, SEED, 0.7, toks[i], stream=streams[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert np.array_equal(toks[i].cpu().numpy(), refs[i])
    tok = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.biv_gumbel_argmax(xd[0], rq, ps, SEED, 0.7, tok, stream=s)     # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.biv_gumbel_argmax(xd[1], rq, ps, SEED, 0.7, tok, stream=torch.cuda.current_stream())
    for _ in range(4):
        tok.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), refs[1])
    # the workspace entry: one workspace per stream, back-to-back launches on two
    # streams at once, then graph replays
    wss = [torch.empty(B.biv_gumbel_argmax_workspace_size(R, V), dtype=torch.uint8, device="cuda")
           for _ in range(2)]
    for _ in range(3):
        for i in range(2):
            toks[i].fill_(-7)
        torch.cuda.synchronize()
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                for _ in range(3):
                    B.biv_gumbel_argmax_ws(xd[i], rq, ps, SEED, 0.7, toks[i], wss[i], stream=streams[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert np.array_equal(toks[i].cpu().numpy(), refs[i])
    graph_ws = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ws):
        B.biv_gumbel_argmax_ws(xd[0], rq, ps, SEED, 0.7, tok, wss[0], stream=torch.cuda.current_stream())
    for _ in range(3):
        tok.fill_(-7)
        graph_ws.replay()
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), refs[0])


def test_gumbel_argmax_chi_square_counts_match_oracle():
    # the 10^6-draw sampling check of the oracle, repeated on the GPU: identical tokens
    x = np.array([0.5, -1.0, 2.0, 0.0, 1.0, -0.5, 1.5, 0.3], np.float32)
    n = 1_000_000
    logits = torch.tensor(np.broadcast_to(x, (n, 8)).copy())
    idx = np.arange(n)
    req, pos = (idx // 1000).astype(np.int32), (idx % 1000).astype(np.int32)
    tok = torch.empty(n, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(logits.cuda(), i32(req), i32(pos), SEED, 1.0, tok)
    ref = oracle.gumbel_argmax(logits, req, pos, SEED, 1.0)
    assert np.array_equal(tok.cpu().numpy(), ref)


def test_verify_accept_bit_exact():
    rng = np.random.default_rng(0)
    for N, K in ((1, 1), (8, 8), (64, 16), (33, 5)):
        t = rng.integers(0, 10, N * K).astype(np.int32)
        d = np.where(rng.random(N * K) < 0.3, rng.integers(0, 10, N * K), t).astype(np.int32)
        p0 = rng.integers(0, 5000, N).astype(np.int32)
        L = torch.empty(N, dtype=torch.int32, device="cuda")
        nl = torch.empty(N, dtype=torch.int32, device="cuda")
        B.biv_verify_accept(i32(t), i32(d), i32(p0), N, K, L, nl)
        rL, rnl = oracle.verify_accept(t, d, p0, N, K)
        assert np.array_equal(L.cpu().numpy(), rL) and np.array_equal(nl.cpu().numpy(), rnl)


# ------------------------------------------- LM head + selection, fused
def _fused_vs_unfused(A, Bw, T, seed=SEED, write_logits=True):
    M, K = A.shape
    N = Bw.shape[0]
    g = synth.generator(M * 31 + N)
    req = torch.randint(0, 2 ** 31 - 1, (M,), generator=g, dtype=torch.int64).to(torch.int32).cuda()
    pos = torch.randint(0, 100000, (M,), generator=g, dtype=torch.int64).to(torch.int32).cuda()
    ref_logits = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.biv_gemm_nosplitk(A, Bw, ref_logits)
    ref_tok = torch.full((M,), -5, dtype=torch.int32, device="cuda")
    B.biv_gumbel_argmax(ref_logits, req, pos, seed, T, ref_tok)
    ws = torch.empty(max(16, B.biv_lm_head_gumbel_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
    tok = torch.full((M,), -9, dtype=torch.int32, device="cuda")
    logits = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda") if write_logits else None
    B.biv_lm_head_gumbel(A, Bw, req, pos, seed, T, tok, ws, logits=logits)
    torch.cuda.synchronize()
    assert torch.equal(tok, ref_tok)
    if write_logits:
        assert same_bits(logits, ref_logits)
    return tok.cpu().numpy(), ref_logits.cpu(), req.cpu(), pos.cpu()


@pytest.mark.parametrize("M,N,K,T,std", [
    (64, 32000, 1024, 0.7, 0.02), (1, 2048, 256, 1.0, 1.0 / 16), (7, 4104, 192, 0.5, 0.1),
    (130, 5000, 512, 0.7, 0.05), (64, 32000, 1024, 0.0, 0.02), (300, 2056, 136, 2.0, 0.2),
    (16, 152064, 256, 0.7, 0.2), (1000, 8200, 256, 0.7, 0.1), (600, 4104, 320, 0.0, 0.1),
    # CTA pairs with many tiles each: 4 row tiles (each pair keeps its rows, and their
    # best keys from tile to tile) and 3 row tiles (the rows change every tile)
    (1024, 20000, 256, 0.7, 0.05), (600, 32000, 256, 0.7, 0.05),
    # the last, partial wave of pair tiles re-cut into the narrowest tiles one wave
    # holds: 96-column tails (four row pairs, 192-column full tiles, two row pairs),
    # 160 (the 4-row-tile case above), 64 (three row pairs), 128 (an exact fit),
    # 192 and 224 (a partial last row tile); most with a ragged last tail tile
    (1024, 25600, 256, 0.7, 0.05), (1024, 25544, 256, 0.7, 0.05), (1024, 34552, 256, 0.7, 0.05),
    (512, 51088, 256, 0.7, 0.05), (600, 40488, 256, 0.7, 0.05), (300, 9792, 256, 0.7, 0.05),
    (300, 14600, 256, 0.7, 0.05), (300, 17032, 256, 0.7, 0.05)])
def test_lm_head_gumbel_fused_bit_exact(M, N, K, T, std):
    g = synth.generator(M + N + K)
    A = synth.bf16_normal((M, K), 1.0, g).cuda()
    Bw = synth.bf16_normal((N, K), std, g).cuda()
    tok, logits, req, pos = _fused_vs_unfused(A, Bw, T, write_logits=(N * M <= 40_000_000))
    ref = oracle.gumbel_argmax(logits, req, pos, SEED, T)
    assert np.array_equal(tok, ref)


@pytest.mark.parametrize("M", [48, 300])          # one CTA per 128-row tile / CTA pairs
def test_lm_head_gumbel_fused_peaked_ties_and_nan(M):
    N, K = 8192, 256
    g = synth.generator(4242)
    A = synth.bf16_normal((M, K), 1.0, g)
    Bw = synth.bf16_normal((N, K), 0.05, g)
    # peaked rows: B row 777 aligned with A row 0, row 5000 with A row 1
    Bw[777] = A[0] * 0.5
    Bw[5000] = A[1] * 0.5
    # exact ties: two identical B rows give identical logits in every row
    Bw[123] = Bw[4000]
    Bw[6001] = Bw[6000]
    # a NaN column (never wins) and an all-NaN row (selects 0)
    Bw[2500, 3] = float("nan")
    A[7] = float("nan")
    A, Bw = A.cuda(), Bw.cuda()
    for T in (0.0, 0.7, 1e-3):
        tok, logits, req, pos = _fused_vs_unfused(A, Bw, T)
        assert np.array_equal(tok, oracle.gumbel_argmax(logits, req, pos, SEED, T))
        assert tok[7] == 0
        assert np.all(tok != 2500)
        if T == 0.0:
            assert tok[0] == 777 and tok[1] == 5000


@pytest.mark.parametrize("n_req,K", [(8, 8), (3, 5), (1, 1), (37, 4)])
def test_lm_head_gumbel_accept_equals_two_calls(n_req, K):
    """LM head + winners/accept in one kernel: tokens, accept lengths and new
    lengths bit-identical to biv_lm_head_gumbel then biv_verify_accept, and
    the accept the oracle computes from the oracle's tokens."""
    M, N, Kd = n_req * K, 4096, 256
    g = synth.generator(n_req * 100 + K)
    A = synth.bf16_normal((M, Kd), 1.0, g).cuda()
    Bw = synth.bf16_normal((N, Kd), 0.1, g).cuda()
    req = torch.arange(M, dtype=torch.int32, device="cuda") // K * 11 + 5
    pos = (torch.arange(M, dtype=torch.int32, device="cuda") % K) + 300
    p0 = torch.arange(n_req, dtype=torch.int32) * 7 + 300
    ws = torch.empty(B.biv_lm_head_gumbel_workspace_size(M, N, Kd), dtype=torch.uint8, device="cuda")
    tok = torch.empty(M, dtype=torch.int32, device="cuda")
    logits = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.biv_lm_head_gumbel(A, Bw, req, pos, SEED, 0.7, tok, ws, logits=logits)
    # drafts: the targets with every third row wrong
    draft = tok.clone()
    draft[::3] = (draft[::3] + 1) % N
    L2, n2 = (torch.empty(n_req, dtype=torch.int32, device="cuda") for _ in range(2))
    B.biv_verify_accept(tok, draft, p0.cuda(), n_req, K, L2, n2)
    tok1 = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    L1, n1 = (torch.full((n_req,), -1, dtype=torch.int32, device="cuda") for _ in range(2))
    B.biv_lm_head_gumbel_accept(A, Bw, req, pos, SEED, 0.7, tok1, draft, p0.cuda(), n_req, K, L1, n1, ws)
    assert torch.equal(tok1, tok) and torch.equal(L1, L2) and torch.equal(n1, n2)
    ref_tok = oracle.gumbel_argmax(logits.cpu(), req.cpu(), pos.cpu(), SEED, 0.7)
    assert np.array_equal(tok1.cpu().numpy(), ref_tok)
    rL, rn = oracle.verify_accept(ref_tok, draft.cpu(), p0, n_req, K)
    assert np.array_equal(L1.cpu().numpy(), rL) and np.array_equal(n1.cpu().numpy(), rn)


def test_lm_head_gumbel_rows_invariant_across_M():
    N, K = 32000, 1024
    g = synth.generator(99)
    A = synth.bf16_normal((256, K), 1.0, g).cuda()
    Bw = synth.bf16_normal((N, K), 0.02, g).cuda()
    req = torch.arange(256, dtype=torch.int32, device="cuda") * 3 + 1
    pos = torch.arange(256, dtype=torch.int32, device="cuda") + 500
    outs = {}
    for M in (1, 8, 64, 129, 256):
        ws = torch.empty(B.biv_lm_head_gumbel_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
        tok = torch.empty(M, dtype=torch.int32, device="cuda")
        B.biv_lm_head_gumbel(A[:M], Bw, req[:M], pos[:M], SEED, 0.7, tok, ws)
        outs[M] = tok.cpu()
    for M, t in outs.items():
        assert torch.equal(t, outs[256][:M]), M
