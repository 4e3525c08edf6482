"""Pins for the oracle's dense stages (CPU only): closed forms, invariants,
special cases that reduce to numpy/scipy routines, and brute force on tiny
inputs.  A dropped term, a wrong sign or index, or a transposed operand in
the oracle fails at least one of these.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from invariant_verify_gb300 import synth


def bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


# --------------------------------------------------------------- bf16 I/O
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.normal(0, 10, 100_000).astype(np.float32)
    ours = oracle.to_bf16(x.astype(np.float64))
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # Ties go to even; a value just above a tie goes up even if fp32 cannot hold it.
    one = 1.0
    assert oracle.to_bf16([one + 2.0 ** -8])[0] == 0x3F80            # tie -> even (1.0)
    assert oracle.to_bf16([one + 3 * 2.0 ** -8])[0] == 0x3F82        # tie -> even (up)
    assert oracle.to_bf16([one + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81
    assert np.array_equal(oracle.from_bf16(ours), torch.tensor(x).to(torch.bfloat16).double().numpy())


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row():
    d, eps = 64, 1e-6
    w = np.linspace(-2, 2, d)
    for c in (1.0, -3.5, 1e-3):
        y = oracle.rmsnorm(np.full((1, d), c), w, eps)
        assert np.allclose(y[0], c / math.sqrt(c * c + eps) * w, rtol=1e-14, atol=0)


def test_rmsnorm_one_hot_row():
    d, eps, a = 256, 1e-6, 5.0
    x = np.zeros((3, d))
    x[0, 7] = a
    x[1, 0] = -a
    x[2, d - 1] = a
    w = np.arange(1, d + 1, dtype=np.float64)
    y = oracle.rmsnorm(x, w, eps)
    val = a / math.sqrt(a * a / d + eps)
    assert math.isclose(y[0, 7], val * w[7], rel_tol=1e-14)
    assert math.isclose(y[1, 0], -val * w[0], rel_tol=1e-14)
    assert math.isclose(y[2, d - 1], val * w[d - 1], rel_tol=1e-14)
    assert np.count_nonzero(y) == 3


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 1024))
    y1 = oracle.rmsnorm(x, np.ones(1024), 1e-12)
    y2 = oracle.rmsnorm(37.0 * x, np.ones(1024), 1e-12)
    assert np.allclose(y1, y2, rtol=1e-10)
    assert np.allclose(np.sqrt((y1 ** 2).mean(axis=1)), 1.0, rtol=1e-10)


# --------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(1, 64, 128), (3, 64, 128), (17, 48, 256)])
def test_gemm_matches_numpy_fp64(M, N, K):
    g = synth.generator(M * 1000 + N)
    A = synth.bf16_normal((M, K), 1.0, g)
    B = synth.bf16_normal((N, K), 0.05, g)
    ref = A.double().numpy() @ B.double().numpy().T
    assert np.allclose(oracle.gemm(A, B), ref, rtol=1e-12, atol=1e-12)


def test_gemm_identity_permutation_and_one_hot():
    K = 64
    A = synth.bf16_normal((5, K), 1.0, synth.generator(9))
    perm = np.random.default_rng(2).permutation(K)
    B = bf16(np.eye(K)[perm])                 # row n picks column perm[n] of A
    C = oracle.gemm(A, B)
    assert np.array_equal(C, A.double().numpy()[:, perm])
    onehot = np.zeros((1, K))
    onehot[0, 11] = 1.0
    Bw = synth.bf16_normal((7, K), 1.0, synth.generator(10))
    assert np.array_equal(oracle.gemm(onehot, Bw)[0], Bw.double().numpy()[:, 11])


def test_gemm_sampled_equals_full():
    A = synth.bf16_normal((9, 96), 1.0, synth.generator(11))
    B = synth.bf16_normal((33, 96), 1.0, synth.generator(12))
    full = oracle.gemm(A, B)
    m = np.array([0, 8, 4, 3]); n = np.array([32, 0, 17, 5])
    assert np.array_equal(oracle.gemm_sampled(A, B, m, n), full[m, n])


# --------------------------------------------------------------- attention
def _cache(n_slots, Hkv, max_len, hd, seed, std=1.0):
    g = synth.generator(seed)
    t = synth.bf16_normal((n_slots, Hkv, max_len, hd), std, g)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_attention_first_position_returns_v0():
    hd, Hq, Hkv = 128, 4, 2
    kc, vc = _cache(2, Hkv, 16, hd, 1), _cache(2, Hkv, 16, hd, 2)
    q = np.random.default_rng(0).normal(size=(2, Hq, hd))
    o = oracle.attention(q, kc, vc, [1, 0], [0, 0])
    v = oracle.from_bf16(vc)
    for w, slot in enumerate([1, 0]):
        for h in range(Hq):
            assert np.array_equal(o[w, h], v[slot, h // 2, 0])


def test_attention_equal_keys_average_values():
    hd, p = 128, 300
    kc = np.zeros((1, 1, 512, hd), np.uint16)
    kc[...] = oracle.to_bf16(np.full(hd, 0.25))              # every key identical
    vc = _cache(1, 1, 512, hd, 3)
    q = np.random.default_rng(1).normal(size=(1, 1, hd))
    o = oracle.attention(q, kc, vc, [0], [p])
    assert np.allclose(o[0, 0], oracle.from_bf16(vc)[0, 0, : p + 1].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # q = a e_0, k_0 = b e_0, k_1 = 0, v_0 = 1, v_1 = 0: o = sigmoid(a b / sqrt(hd)).
    hd, a, b = 128, 3.0, 2.0
    kc = np.zeros((1, 1, 4, hd), np.uint16); vc = np.zeros_like(kc)
    kc[0, 0, 0, 0] = oracle.to_bf16([b])[0]
    vc[0, 0, 0, :] = oracle.to_bf16(np.ones(hd))
    q = np.zeros((1, 1, hd)); q[0, 0, 0] = a
    o = oracle.attention(q, kc, vc, [0], [1])
    assert np.allclose(o[0, 0], 1.0 / (1.0 + math.exp(-a * b / math.sqrt(hd))), rtol=1e-14)


def test_attention_gqa_head_mapping():
    # Query head h reads KV head h // (Hq/Hkv): give each KV head constant values.
    hd, Hq, Hkv = 128, 8, 2
    kc = _cache(1, Hkv, 8, hd, 4)
    vc = np.zeros((1, Hkv, 8, hd), np.uint16)
    for h in range(Hkv):
        vc[0, h] = oracle.to_bf16(np.full((8, hd), h + 1.0))
    q = np.random.default_rng(2).normal(size=(1, Hq, hd))
    o = oracle.attention(q, kc, vc, [0], [5])
    for h in range(Hq):
        assert np.allclose(o[0, h], h // (Hq // Hkv) + 1.0, rtol=1e-14)


@pytest.mark.parametrize("p", [255, 256, 257, 511, 512])
def test_attention_brute_force_at_split_boundaries(p):
    hd, Hq, Hkv = 128, 4, 2
    kc, vc = _cache(1, Hkv, 640, hd, 5), _cache(1, Hkv, 640, hd, 6)
    q = np.random.default_rng(p).normal(size=(1, Hq, hd))
    o = oracle.attention(q, kc, vc, [0], [p])
    K, V = oracle.from_bf16(kc), oracle.from_bf16(vc)
    for h in range(Hq):
        s = K[0, h // 2, : p + 1] @ q[0, h] / math.sqrt(hd)
        ref = softmax(s) @ V[0, h // 2, : p + 1]
        assert np.allclose(o[0, h], ref, rtol=1e-11, atol=1e-13)
    # The sampled variant agrees with the full one.
    qb = oracle.to_bf16(q)
    full = oracle.attention(oracle.from_bf16(qb), kc, vc, [0], [p])
    samp = oracle.attention_sampled(qb.reshape(1, Hq, hd), kc, vc, [0], [p], [0, 0], [3, 1])
    assert np.allclose(samp, full[0, [3, 1]], rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity_and_norm_preserving():
    x = np.random.default_rng(3).normal(size=(4, 3, 128))
    assert np.array_equal(oracle.rope(x, [0, 0, 0, 0], 10000.0), x)
    y = oracle.rope(x, [1, 17, 400, 4095], 500000.0)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_first_pair_rotates_by_position():
    # Pair (0, hd/2) has frequency theta^0 = 1: angle = pos radians.
    x = np.zeros((1, 1, 128)); x[0, 0, 0] = 1.0
    for pos in (1, 5, 1000):
        y = oracle.rope(x, [pos], 10000.0)
        assert math.isclose(y[0, 0, 0], math.cos(pos), abs_tol=1e-14)
        assert math.isclose(y[0, 0, 64], math.sin(pos), abs_tol=1e-14)
    # Pair i has frequency theta^(-2i/hd): pick i = 32 -> theta^(-1/2).
    x = np.zeros((1, 1, 128)); x[0, 0, 32] = 1.0
    y = oracle.rope(x, [100], 10000.0)
    assert math.isclose(y[0, 0, 96], math.sin(100 / 100.0), abs_tol=1e-14)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=(1, 1, 128)), rng.normal(size=(1, 1, 128))
    s = [float(oracle.rope(q, [a + 7], 500000.0)[0, 0] @ oracle.rope(k, [a], 500000.0)[0, 0])
         for a in (0, 100, 3000)]
    assert np.allclose(s, s[0], rtol=1e-10)


# ------------------------------------------------------------------ SwiGLU
def test_silu_mul_closed_forms():
    gu = np.array([[0.0, 1.0, 40.0, -40.0, 3.0, 2.0, 5.0, 7.0]])   # F = 4
    h = oracle.silu_mul(gu)[0]
    assert h[0] == 0.0
    assert math.isclose(h[1], 1.0 / (1.0 + math.exp(-1.0)) * 2.0, rel_tol=1e-15)
    assert math.isclose(h[2], 40.0 * 5.0, rel_tol=1e-15)
    assert math.isclose(h[3], -40.0 * 7.0 / (1.0 + math.exp(40.0)), rel_tol=1e-12)   # ~ -1.2e-15


# ---------------------------------------------------------------- KV write
def test_kv_overwrite_writes_only_the_window_rows():
    kc = _cache(3, 2, 32, 128, 7); vc = _cache(3, 2, 32, 128, 8)
    k0, v0 = kc.copy(), vc.copy()
    kn = _cache(1, 4, 2, 128, 9).reshape(4, 2, 128)
    vn = _cache(1, 4, 2, 128, 10).reshape(4, 2, 128)
    slots, pos = np.array([2, 2, 0, 1]), np.array([5, 6, 31, 0])
    oracle.kv_overwrite(kc, vc, kn, vn, slots, pos)
    for w in range(4):
        assert np.array_equal(kc[slots[w], :, pos[w]], kn[w])
        assert np.array_equal(vc[slots[w], :, pos[w]], vn[w])
        k0[slots[w], :, pos[w]] = kn[w]; v0[slots[w], :, pos[w]] = vn[w]
    assert np.array_equal(kc, k0) and np.array_equal(vc, v0)


def test_random_bf16_rounding_picks_a_bracketing_value():
    """round_bf16_random returns, for every element, one of the two bf16
    values that bracket it (the value itself if bf16 holds it exactly), each
    side about half the time: the grid is rebuilt here from frexp, not from
    the oracle's bf16 conversion."""
    rng = np.random.default_rng(3)
    n = 40000
    x = rng.normal(size=n) * 10.0 ** rng.integers(-30, 30, n)
    exact = np.array([0.0, -0.0, 1.0, -2.5, 0.15625, 2.0 ** 127, -1.0 / 1024, 3.0 * 2.0 ** -100])
    x = np.concatenate([x, exact])
    y = oracle.round_bf16_random(x, np.random.default_rng(4))
    m, e = np.frexp(x)                     # |x| = |m| 2^e, 0.5 <= |m| < 1
    sp = np.ldexp(1.0, e - 8)              # bf16 spacing: 8 significant bits
    lo, hi = np.floor(x / sp) * sp, np.ceil(x / sp) * sp
    assert np.all((y == lo) | (y == hi))
    assert np.array_equal(y[-len(exact):], exact)
    inexact = lo[:n] != hi[:n]
    up = (y[:n] == hi[:n]) & inexact
    frac_up = up.sum() / inexact.sum()
    assert 0.48 < frac_up < 0.52, frac_up
    # the nearest-rounding oracle picks the nearer of the same two values
    near = oracle.round_bf16(x[:n])
    assert np.all((near == lo[:n]) | (near == hi[:n]))
    assert np.all(np.abs(near - x[:n]) <= np.abs(np.where(near == lo[:n], hi[:n], lo[:n]) - x[:n]))
