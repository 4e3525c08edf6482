"""Pins for the Gumbel top-k selection and the n-gram lookup drafter (CPU).

* Gumbel top-k (AIexTime post 185: the Gumbel-max trick gives top-k
  sampling as it stands; Kool et al., "Stochastic Beams and Where to Find
  Them"): the k largest keys, in order, are k draws without replacement from
  softmax(x / T), so the first two positions follow the Plackett-Luce law
  P(i, j) = p_i p_j / (1 - p_i); at T = 0 the order is the sorted logits.
* n-gram drafter (NVIDIA inference guide page: a training-free method that
  finds and copies repeated fragments of the earlier text): on a periodic
  history the drafts continue the period; the copied run always follows a
  real occurrence of the history's suffix, of the longest available n, at the
  most recent position, and a run that reaches the end of the history
  continues from its own output.
"""
import numpy as np
import pytest

import oracle

SEED = 0x1234_5678_9ABC_DEF0


# ---------------------------------------------------------------- top-k
def _topk_numpy(x, req, pos, T, k):
    """Independent ordering: numpy lexsort of (-key, index) over the oracle's noise."""
    out = []
    invT = np.float32(1.0) / np.float32(T) if T > 0 else np.float32(0)
    for r in range(x.shape[0]):
        if T > 0:
            g = oracle.gumbel_row(SEED, int(req[r]), int(pos[r]) + 1, x.shape[1])
            key = (x[r] * invT).astype(np.float32) + g
        else:
            key = x[r]
        order = np.lexsort((np.arange(x.shape[1]), -key.astype(np.float64)))
        out.append(order[:k])
    return np.array(out, np.int32)


@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_topk_is_the_sorted_keys(T):
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, (20, 300)).astype(np.float32)
    x[3, 10] = x[3, 200] = x[3].max() + 1      # an exact tie at the top
    req = rng.integers(0, 2 ** 31 - 1, 20)
    pos = rng.integers(0, 5000, 20).astype(np.int32)
    got = oracle.gumbel_topk(x, req, pos, SEED, T, 12)
    assert np.array_equal(got, _topk_numpy(x, req, pos, T, 12))
    assert np.array_equal(got[:, 0], oracle.gumbel_argmax(x, req, pos, SEED, T))
    assert all(len(set(row)) == 12 for row in got)
    if T == 0.0:
        assert got[3, 0] == 10 and got[3, 1] == 200


def test_topk_full_permutation_and_k1():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (5, 17)).astype(np.float32)
    req = np.arange(5)
    pos = np.arange(5, dtype=np.int32)
    full = oracle.gumbel_topk(x, req, pos, SEED, 1.0, 17)
    assert all(sorted(r) == list(range(17)) for r in full)
    assert np.array_equal(oracle.gumbel_topk(x, req, pos, SEED, 1.0, 1)[:, 0], full[:, 0])


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_topk_first_two_follow_plackett_luce(T):
    # chi-square over the 12 ordered pairs (11 dof, alpha = 1e-3 -> 31.26)
    logits = np.array([0.3, -0.5, 1.1, 0.0], np.float32)
    n = 200_000
    x = np.tile(logits, (n, 1))
    req = np.arange(n) % 977 + 5
    pos = (np.arange(n) // 977).astype(np.int32) * 3 + 11
    top = oracle.gumbel_topk(x, req, pos, SEED, T, 2)
    z = logits.astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    chi2 = 0.0
    for i in range(4):
        for j in range(4):
            if i == j:
                continue
            e = n * p[i] * p[j] / (1 - p[i])
            o = np.count_nonzero((top[:, 0] == i) & (top[:, 1] == j))
            chi2 += (o - e) ** 2 / e
    assert chi2 < 31.26, chi2


# --------------------------------------------------------------- n-gram
def test_ngram_worked_example():
    # history 5 7 1 2 3 4 9 1 2 3: the suffix "1 2 3" occurred at position 2,
    # followed by 4 9 1 2 3 -> drafts 4 9 1 2 (K = 4)
    h = np.array([[5, 7, 1, 2, 3, 4, 9, 1, 2, 3]], np.int32)
    d, src = oracle.ngram_draft(h, [10], 3, 1, 4)
    assert d.tolist() == [[4, 9, 1, 2]] and src.tolist() == [5]


def test_ngram_continues_a_period():
    for period in (2, 3, 5, 7):
        pat = np.arange(period, dtype=np.int32) * 11 + 3
        h = np.tile(pat, 200 // period + 1)[None, :].astype(np.int32)
        for L in (period * 3, period * 3 + 1, 97):
            d, _ = oracle.ngram_draft(h, [L], 4, 1, 8)
            assert d[0].tolist() == [int(pat[(L + j) % period]) for j in range(8)], (period, L)


def test_ngram_short_and_missing():
    h = np.array([[4, 0, 0], [6, 6, 0], [1, 2, 3], [0, 0, 0]], np.int32)
    d, src = oracle.ngram_draft(h, [1, 2, 3, 0], 2, 1, 3)
    assert d[0].tolist() == [4, 4, 4] and src[0] == -1        # nothing to match
    assert d[1].tolist() == [6, 6, 6] and src[1] == 1          # "6" then 6, continued from the copy
    assert d[2].tolist() == [3, 3, 3] and src[2] == -1         # no repeat: the last token
    assert d[3].tolist() == [0, 0, 0] and src[3] == -1         # empty history


def test_ngram_choice_is_longest_then_latest():
    rng = np.random.default_rng(8)
    N, ld = 300, 120
    h = rng.integers(0, 4, (N, ld)).astype(np.int32)      # small alphabet: many repeats
    lens = rng.integers(0, ld + 1, N).astype(np.int32)
    n_max, n_min, K = 4, 2, 6
    d, src = oracle.ngram_draft(h, lens, n_max, n_min, K)
    for r in range(N):
        L = int(lens[r])
        hr = h[r, :L]
        found = None
        for n in range(n_max, n_min - 1, -1):
            if L < n + 1:
                continue
            suf = hr[L - n:]
            ps = [p for p in range(L - n) if np.array_equal(hr[p:p + n], suf)]
            if ps:
                found = (n, max(ps))
                break
        if found is None:
            assert src[r] == -1
            assert (d[r] == (hr[-1] if L else 0)).all()
            continue
        n, p = found
        assert src[r] == p + n
        ext = hr.tolist()
        for j in range(K):                  # copy with overlap: the run may read its own output
            ext.append(ext[p + n + j])
        assert d[r].tolist() == ext[L:]
