"""CPU oracle for the batch-invariant verification step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It never touches CUDA and shares no code with
the GPU library: the arithmetic lives in ``oracle.cpp`` (plain C++, fp64 for
the dense parts, the exact fp32 rule for selection) and this module only
marshals numpy arrays into it.

Functions without an independent pin are marked "parity unpinned" in their
docstring.  (Currently none: every entry point is pinned by a closed form,
a published test vector, a brute-force / library special case or a
statistical property in ``tests/test_oracle_*.py``.)
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, f32, f64, u32, u64 = C.c_int, C.c_longlong, C.c_float, C.c_double, C.c_uint32, C.c_uint64
        sig = {
            "orc_num_threads": (i32, []),
            "orc_set_threads": (None, [i32]),
            "orc_bf16_to_f64": (None, [P, i64, P]),
            "orc_f64_to_bf16": (None, [P, i64, P]),
            "orc_rmsnorm": (None, [P, P, i32, i32, f64, P]),
            "orc_gemm": (None, [P, P, i32, i32, i32, P]),
            "orc_gemm_sampled": (None, [P, P, i32, P, P, i32, P]),
            "orc_rope": (None, [P, P, i32, i32, i32, f64]),
            "orc_attention": (None, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]),
            "orc_attention_sampled": (None, [P, P, P, P, P, i32, i32, i32, i32, P, P, i32, P]),
            "orc_silu_mul": (None, [P, i32, i32, P]),
            "orc_kv_overwrite": (None, [P, P, P, P, P, P, i32, i32, i32, i32]),
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_uniform": (f32, [u32]),
            "orc_log_f32": (f32, [f32]),
            "orc_log_batch": (None, [P, i64, P]),
            "orc_gumbel_from_word": (f32, [u32]),
            "orc_gumbel_from_words": (None, [P, i64, P]),
            "orc_gumbel": (f32, [u64, u32, u32, u32]),
            "orc_gumbel_row": (None, [u64, u32, u32, i32, P]),
            "orc_gumbel_argmax": (None, [P, i32, i32, i64, P, P, u64, f32, P]),
            "orc_verify_accept": (None, [P, P, P, i32, i32, P, P]),
            "orc_gumbel_topk": (None, [P, i32, i32, i64, P, P, u64, f32, i32, P]),
            "orc_ngram_draft": (None, [P, i32, i64, P, i32, i32, i32, P, P]),
            "orc_gqa_max_drafts": (i32, [i32, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers
def _np(x, dtype=None):
    """torch tensor or array-like -> contiguous numpy array (bf16 -> uint16 bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x if dtype is None else np.asarray(x, dtype=dtype))
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def from_bf16(x) -> np.ndarray:
    a = _np(x)
    assert a.dtype == np.uint16, a.dtype
    out = np.empty(a.shape, np.float64)
    lib().orc_bf16_to_f64(_p(a), a.size, _p(out))
    return out


def to_bf16(x) -> np.ndarray:
    a = _np(x, np.float64)
    out = np.empty(a.shape, np.uint16)
    lib().orc_f64_to_bf16(_p(a), a.size, _p(out))
    return out


def round_bf16(x) -> np.ndarray:
    """fp64 values rounded to the nearest bf16 and returned as fp64."""
    return from_bf16(to_bf16(x))


def round_bf16_random(x, rng) -> np.ndarray:
    """fp64 values rounded to one of their two bracketing bf16 values, chosen
    at random (``rng``: a numpy Generator), returned as fp64; values a bf16
    holds exactly are unchanged.

    Any correct bf16 implementation stores, at each storage point, the
    nearest bf16 of a value within a few fp32 ulps of the exact one, so it
    differs from the nearest-bf16 oracle by at most one bf16 ulp per stored
    element.  A composition that rounds every stored element in a random
    direction departs from the oracle by up to one ulp at (about half of) all
    elements of every storage point, an envelope for that drift; the
    end-to-end GPU tests take their logit tolerance from it."""
    a = _f64(x)
    near = to_bf16(a)                               # nearest bf16 (ties to even)
    nv = from_bf16(near)
    # the other bracketing bf16: one step away from `near`, towards x
    away = np.abs(a) > np.abs(nv)                   # x lies beyond `near` in magnitude
    other = near.astype(np.int32) + np.where(away, 1, -1)
    zero_mag = (near & 0x7FFF) == 0
    other = np.where(zero_mag & (a != nv), (np.signbit(a).astype(np.int32) << 15) | 1, other)
    other = (other & 0xFFFF).astype(np.uint16)
    ov = from_bf16(other)
    pick = rng.random(a.shape) < 0.5
    return np.where((a != nv) & pick, ov, nv)


def _f64(x) -> np.ndarray:
    a = _np(x)
    if a.dtype == np.uint16:
        return from_bf16(a)
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------- kernels
def rmsnorm(x, w, eps: float) -> np.ndarray:
    xd, wd = _f64(x), _f64(w)
    rows, d = xd.shape
    y = np.empty_like(xd)
    lib().orc_rmsnorm(_p(xd), _p(wd), rows, d, float(eps), _p(y))
    return y


def gemm(A, B) -> np.ndarray:
    """C = A @ B^T in fp64; A fp64 or bf16 [M,K], B bf16 [N,K]."""
    Ad = _f64(A)
    Bb = _np(B)
    assert Bb.dtype == np.uint16
    M, K = Ad.shape
    N = Bb.shape[0]
    assert Bb.shape[1] == K
    out = np.empty((M, N), np.float64)
    lib().orc_gemm(_p(Ad), _p(Bb), M, N, K, _p(out))
    return out


def gemm_sampled(A, B, m_idx, n_idx) -> np.ndarray:
    Ab, Bb = _np(A), _np(B)
    assert Ab.dtype == np.uint16 and Bb.dtype == np.uint16
    mi = np.ascontiguousarray(m_idx, np.int64)
    ni = np.ascontiguousarray(n_idx, np.int64)
    out = np.empty(mi.size, np.float64)
    lib().orc_gemm_sampled(_p(Ab), _p(Bb), Ab.shape[1], _p(mi), _p(ni), mi.size, _p(out))
    return out


def rope(x, row_pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [rows, heads, hd] at the rows' positions (copy)."""
    xd = _f64(x).copy()
    rows, heads, hd = xd.shape
    pos = np.ascontiguousarray(row_pos, np.int32)
    lib().orc_rope(_p(xd), _p(pos), rows, heads, hd, float(theta))
    return xd


def attention(q, k_cache, v_cache, row_slot, row_pos) -> np.ndarray:
    qd = _f64(q)
    W, Hq, hd = qd.shape
    kc, vc = _np(k_cache), _np(v_cache)
    n_slots, Hkv, max_len, hd2 = kc.shape
    assert hd2 == hd and kc.dtype == np.uint16
    rs = np.ascontiguousarray(row_slot, np.int32)
    rp = np.ascontiguousarray(row_pos, np.int32)
    assert (rp < max_len).all() and (rp >= 0).all()
    o = np.empty_like(qd)
    lib().orc_attention(_p(qd), _p(kc), _p(vc), _p(rs), _p(rp), W, Hq, Hkv, hd, n_slots, max_len, _p(o))
    return o


def attention_sampled(q_bf16, k_cache, v_cache, row_slot, row_pos, rows, heads) -> np.ndarray:
    qb = _np(q_bf16)
    W, Hq, hd = qb.shape
    kc, vc = _np(k_cache), _np(v_cache)
    _, Hkv, max_len, _ = kc.shape
    rs = np.ascontiguousarray(row_slot, np.int32)
    rp = np.ascontiguousarray(row_pos, np.int32)
    ri = np.ascontiguousarray(rows, np.int32)
    hi = np.ascontiguousarray(heads, np.int32)
    o = np.empty((ri.size, hd), np.float64)
    lib().orc_attention_sampled(_p(qb), _p(kc), _p(vc), _p(rs), _p(rp), Hq, Hkv, hd, max_len,
                                _p(ri), _p(hi), ri.size, _p(o))
    return o


def silu_mul(gu) -> np.ndarray:
    g = _f64(gu)
    rows, two_f = g.shape
    out = np.empty((rows, two_f // 2), np.float64)
    lib().orc_silu_mul(_p(g), rows, two_f // 2, _p(out))
    return out


def kv_overwrite(k_cache: np.ndarray, v_cache: np.ndarray, k_new, v_new, row_slot, row_pos) -> None:
    """In-place write of the window's K/V rows (all uint16 bf16 arrays)."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    kn, vn = _np(k_new), _np(v_new)
    W, Hkv, hd = kn.shape
    rs = np.ascontiguousarray(row_slot, np.int32)
    rp = np.ascontiguousarray(row_pos, np.int32)
    max_len = k_cache.shape[2]
    assert (rp < max_len).all()
    lib().orc_kv_overwrite(_p(k_cache), _p(v_cache), _p(kn), _p(vn), _p(rs), _p(rp), W, Hkv, hd, max_len)


# -------------------------------------------------------------- selection
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform(w: int) -> float:
    return lib().orc_uniform(int(w) & 0xFFFFFFFF)


def log_f32(x) -> np.ndarray:
    a = np.ascontiguousarray(x, np.float32)
    out = np.empty_like(a)
    lib().orc_log_batch(_p(a), a.size, _p(out))
    return out


def gumbel_from_words(words) -> np.ndarray:
    w = np.ascontiguousarray(words, np.uint32)
    out = np.empty(w.shape, np.float32)
    lib().orc_gumbel_from_words(_p(w), w.size, _p(out))
    return out


def gumbel(seed: int, req: int, pos: int, v: int) -> float:
    return lib().orc_gumbel(int(seed), int(req) & 0xFFFFFFFF, int(pos) & 0xFFFFFFFF, int(v))


def gumbel_row(seed: int, req: int, pos: int, V: int) -> np.ndarray:
    out = np.empty(V, np.float32)
    lib().orc_gumbel_row(int(seed), int(req) & 0xFFFFFFFF, int(pos) & 0xFFFFFFFF, V, _p(out))
    return out


def gumbel_argmax(logits, row_req, row_pos, seed: int, temperature: float) -> np.ndarray:
    x = _np(logits, np.float32)
    R, V = x.shape
    rq = np.ascontiguousarray(_np(row_req).astype(np.int64) & 0xFFFFFFFF, np.uint32)
    rp = np.ascontiguousarray(_np(row_pos), np.int32)
    out = np.empty(R, np.int32)
    lib().orc_gumbel_argmax(_p(x), R, V, V, _p(rq), _p(rp), int(seed), float(temperature), _p(out))
    return out


def gumbel_keys(logits, row_req, row_pos, seed: int, temperature: float) -> np.ndarray:
    """The selection keys of every entry (fp32 [R, V]): key = fl(fl(x * fl(1/T))
    + g) with g the row's noise at the selected position (row_pos + 1); the
    logits themselves at T = 0.  numpy's fp32 multiply and add are single
    IEEE operations, as the rule requires.  (For tests that look at key gaps.)"""
    x = _np(logits, np.float32).astype(np.float32)
    R, V = x.shape
    if float(temperature) == 0.0:
        return x.copy()
    invT = np.float32(1.0) / np.float32(temperature)
    rq = _np(row_req).astype(np.int64) & 0xFFFFFFFF
    rp = _np(row_pos).astype(np.int64)
    keys = np.empty_like(x)
    for r in range(R):
        g = gumbel_row(seed, int(rq[r]), int(rp[r]) + 1, V)
        keys[r] = (x[r] * invT).astype(np.float32) + g
    return keys


def gumbel_topk(logits, row_req, row_pos, seed: int, temperature: float, k: int) -> np.ndarray:
    """The k largest Gumbel keys of each row, in order (int32 [R, k])."""
    x = _np(logits, np.float32)
    R, V = x.shape
    assert 1 <= k <= V
    rq = np.ascontiguousarray(_np(row_req).astype(np.int64) & 0xFFFFFFFF, np.uint32)
    rp = np.ascontiguousarray(_np(row_pos), np.int32)
    out = np.empty((R, k), np.int32)
    lib().orc_gumbel_topk(_p(x), R, V, V, _p(rq), _p(rp), int(seed), float(temperature), int(k), _p(out))
    return out


def ngram_draft(hist, lengths, n_max: int, n_min: int, K: int):
    """n-gram lookup drafts (int32 [N, K]) and the copy source per request
    (longest n-gram suffix match, most recent occurrence, LZ-style copy)."""
    h = np.ascontiguousarray(_np(hist), np.int32)
    N, ld = h.shape
    ln = np.ascontiguousarray(_np(lengths), np.int32)
    assert ln.shape == (N,) and (ln >= 0).all() and (ln <= ld).all() and 1 <= n_min <= n_max
    d = np.empty((N, K), np.int32)
    src = np.empty(N, np.int32)
    lib().orc_ngram_draft(_p(h), N, ld, _p(ln), int(n_max), int(n_min), int(K), _p(d), _p(src))
    return d, src


def verify_accept(target, draft, p0, N: int, K: int):
    t = np.ascontiguousarray(_np(target), np.int32)
    d = np.ascontiguousarray(_np(draft), np.int32)
    p = np.ascontiguousarray(_np(p0), np.int32)
    assert t.size == N * K and d.size == N * K and p.size == N
    L = np.empty(N, np.int32)
    nl = np.empty(N, np.int32)
    lib().orc_verify_accept(_p(t), _p(d), _p(p), N, K, _p(L), _p(nl))
    return L, nl


def gqa_max_drafts(G: int, tile: int = 128) -> int:
    return lib().orc_gqa_max_drafts(int(G), int(tile))
