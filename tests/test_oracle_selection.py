"""Pins for the oracle's selection rule (CPU only).

Each check ties the oracle to something other than itself: published
Philox test vectors, the fp64 library log, the Gumbel distribution's closed
forms, the softmax the Gumbel-max trick must sample from (tginsight
AIexTime post 185, "Coupling without Communication and Drafter-Invariant
Speculative Decoding": adding Gumbel(0,1) noise and taking the argmax is
equivalent to sampling from the softmax), and numpy's argmax for T = 0.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SEED = 0x1234_5678_9ABC_DEF0


def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(t, 16) for t in line.split()])
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for r in rows:
        out = oracle.philox4x32_10(r[:4], r[4:6])
        assert [int(x) for x in out] == r[6:], [hex(int(x)) for x in out]


def test_uniform_is_exact_and_open():
    # u = (2*(w>>9)+1) * 2^-24: smallest 2^-24, largest 1 - 2^-24, exact dyadics.
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(0x1FF) == 2.0 ** -24           # low 9 bits ignored
    assert oracle.uniform(1 << 31) == 0.5 + 2.0 ** -24
    for w in (12345 << 9, 0xDEADBEEF, 0x80000000):
        k = 2 * (w >> 9) + 1
        assert oracle.uniform(w) == k * 2.0 ** -24


def _all_uniforms():
    k = np.arange(2 ** 23, dtype=np.uint64)
    return ((2 * k + 1).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def _ulp_err(got, ref):
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - ref) / ulp


def test_own_log_exhaustive_within_4ulp():
    u = _all_uniforms()
    assert np.unique(u).size == 2 ** 23
    L = oracle.log_f32(u)
    assert _ulp_err(L, np.log(u.astype(np.float64))).max() <= 4.0
    t = -L                                      # the second log's inputs
    L2 = oracle.log_f32(t)
    ref2 = np.log(t.astype(np.float64))
    nz = ref2 != 0
    assert _ulp_err(L2[nz], ref2[nz]).max() <= 4.0
    assert np.all(L2[~nz] == 0.0)


def test_own_log_special_values():
    x = np.array([1.0, 2.0, 0.5, 4.0, 2.0 ** -24, 16.0, math.e], np.float32)
    L = oracle.log_f32(x)
    assert L[0] == 0.0
    ref = np.log(x.astype(np.float64))
    assert np.all(_ulp_err(L[1:], ref[1:]) <= 1.0)


def test_noise_range_below_pruning_bound():
    # Exhaustive over every uniform the generator can produce: the noise lies in
    # [-2.82, 16.64]; the GPU's exact candidate pruning assumes g < 17.
    k = np.arange(2 ** 23, dtype=np.uint32)
    g = oracle.gumbel_from_words(k << 9)
    assert g.max() < 17.0 and g.max() > 16.6
    assert g.min() > -2.82 and g.min() < -2.8
    # g is a non-decreasing function of u (both logs are monotone here).
    assert np.all(np.diff(g.astype(np.float64)) >= 0)


def test_noise_is_gumbel_distributed():
    # Closed forms of Gumbel(0,1): CDF exp(-exp(-g)), mean = Euler's gamma,
    # variance pi^2/6.  Kolmogorov-Smirnov at alpha = 1e-3 and 5-sigma moments.
    n = 1 << 20
    g = oracle.gumbel_row(SEED, 7, 1234, n).astype(np.float64)
    gs = np.sort(g)
    cdf = np.exp(-np.exp(-gs))
    i = np.arange(1, n + 1)
    D = max(np.max(i / n - cdf), np.max(cdf - (i - 1) / n))
    assert D < 1.95 / math.sqrt(n)
    gamma = 0.5772156649015329
    assert abs(g.mean() - gamma) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 5 * math.sqrt(2.0 * (math.pi ** 2 / 6) ** 2 / n) * 2


def test_noise_counter_layout():
    # One Philox call feeds 4 consecutive vocabulary ids; the noise of v uses
    # output word v & 3 of counter (v >> 2, pos, req, 0) under key = seed.
    req, pos = 11, 777
    row = oracle.gumbel_row(SEED, req, pos, 16)
    for v in range(16):
        words = oracle.philox4x32_10([v >> 2, pos, req, 0], [SEED & 0xFFFFFFFF, SEED >> 32])
        assert oracle.gumbel_from_words(np.array([words[v & 3]], np.uint32))[0] == row[v]
        assert oracle.gumbel(SEED, req, pos, v) == row[v]
    # Different request, position or seed -> different noise.
    assert not np.array_equal(row, oracle.gumbel_row(SEED, req + 1, pos, 16))
    assert not np.array_equal(row, oracle.gumbel_row(SEED, req, pos + 1, 16))
    assert not np.array_equal(row, oracle.gumbel_row(SEED + 1, req, pos, 16))


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_gumbel_max_samples_softmax_chi_square(T):
    # 10^6 draws over distinct (req, pos) counters, V = 8 fixed logits.
    x = np.array([0.5, -1.0, 2.0, 0.0, 1.0, -0.5, 1.5, 0.3], np.float32)
    n = 1_000_000
    logits = np.broadcast_to(x, (n, 8)).copy()
    idx = np.arange(n)
    tokens = oracle.gumbel_argmax(logits, idx // 1000, idx % 1000, SEED, T)
    counts = np.bincount(tokens, minlength=8)
    z = x.astype(np.float64) * np.float64(np.float32(1.0) / np.float32(T))   # softmax(x / T)
    p = np.exp(z - z.max())
    p /= p.sum()
    exp = n * p
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 24.32, (chi2, counts, exp)   # chi^2_7 at alpha = 1e-3


def test_greedy_is_numpy_argmax_with_lowest_index():
    rng = np.random.default_rng(3)
    x = rng.integers(-3, 3, size=(200, 37)).astype(np.float32)   # many exact ties
    tok = oracle.gumbel_argmax(x, np.zeros(200), np.arange(200), SEED, 0.0)
    assert np.array_equal(tok, np.argmax(x, axis=1))


def test_selection_uses_the_output_position():
    # Row at input position p selects the token of position p + 1.
    x = np.zeros((1, 64), np.float32)
    tok = oracle.gumbel_argmax(x, [5], [99], SEED, 1.0)[0]
    g = oracle.gumbel_row(SEED, 5, 100, 64)
    assert tok == int(np.argmax(g))


def test_nan_key_never_wins():
    x = np.array([[np.nan, -50.0, np.nan, -60.0]], np.float32)
    assert oracle.gumbel_argmax(x, [0], [0], SEED, 0.0)[0] == 1
    assert oracle.gumbel_argmax(x, [0], [0], SEED, 1.0)[0] in (1, 3)


def test_peaked_rows_select_the_peak():
    # A logit 100 above the rest beats any noise (noise range is < 20).
    rng = np.random.default_rng(0)
    x = rng.normal(0, 3, size=(64, 1000)).astype(np.float32)
    peak = rng.integers(0, 1000, 64)
    x[np.arange(64), peak] = 100.0
    tok = oracle.gumbel_argmax(x, np.arange(64), np.arange(64), SEED, 0.7)
    assert np.array_equal(tok, peak)


@pytest.mark.parametrize("T", [0.7, 1.0, 0.0])
def test_gumbel_keys_argmax_is_the_selection(T):
    """The per-entry keys the end-to-end tests use for key gaps: their
    first largest entry is the oracle's selected token on every row."""
    g = np.random.default_rng(17)
    R, V = 24, 3000
    x = (g.normal(size=(R, V)) * 3.0).astype(np.float32)
    x[::5, 7] = x[::5].max(axis=1) + 0.01              # near-peaked rows
    req = g.integers(0, 2 ** 31 - 1, R)
    pos = g.integers(0, 100000, R).astype(np.int32)
    keys = oracle.gumbel_keys(x, req, pos, SEED, T)
    tok = oracle.gumbel_argmax(x, req, pos, SEED, T)
    assert np.array_equal(np.argmax(keys, axis=1), tok)
