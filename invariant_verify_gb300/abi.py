"""Thin ctypes binding of libbiv (``include/biv.h``), same names as the C ABI.

Each ``biv_*`` function takes torch CUDA tensors, passes their raw device
pointers, sizes and the current CUDA stream to the C entry point of the same
name, and raises ``BivError`` on a non-zero status.  There is no fallback:
if ``libbiv.so`` has not been built, loading raises immediately.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbiv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "biv.h")

BIV_BF16, BIV_F32 = 0, 1
KV_SPLIT, HEAD_DIM, ATTN_TILE = 256, 128, 128
NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None


class BivError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _load().biv_status_string(status).decode()
        extra = ""
        if status == 6:
            extra = f" (cudaError {_load().biv_last_cuda_error()})"
        super().__init__(f"{fn}: status {status}: {msg}{extra}")
        self.status = status


_P, _I, _LL, _F, _U64, _SZ = C.c_void_p, C.c_int, C.c_longlong, C.c_float, C.c_uint64, C.c_size_t
SIGNATURES = {
    "biv_status_string": (C.c_char_p, [_I]),
    "biv_last_cuda_error": (_I, []),
    "biv_version": (_I, []),
    "biv_device_error": (_I, [_P]),
    "biv_selftest_wait_timeout": (_I, [_P]),
    "biv_rmsnorm": (_I, [_P, _P, _P, _I, _I, _F, _P]),
    "biv_gemm_nosplitk": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "biv_gemm_nosplitk_bn": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "biv_gemm_tile_n": (_I, [_I, _I, _I]),
    "biv_decode_attn_workspace_size": (_SZ, [_I, _I, _I]),
    "biv_decode_attn_fixedsplit": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "biv_decode_attn_fixedsplit_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "biv_gqa_max_drafts": (_I, [_I, _I]),
    "biv_kv_overwrite": (_I, [_P, _P, _P, _LL, _P, _LL, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "biv_gumbel_argmax": (_I, [_P, _I, _I, _LL, _P, _P, _U64, _F, _P, _P]),
    "biv_gumbel_argmax_workspace_size": (_SZ, [_I, _I]),
    "biv_gumbel_argmax_ws": (_I, [_P, _I, _I, _LL, _P, _P, _U64, _F, _P, _P, _SZ, _P]),
    "biv_gumbel_noise": (_I, [_U64, _P, _P, _I, _I, _P, _P]),
    "biv_gumbel_topk": (_I, [_P, _I, _I, _LL, _P, _P, _U64, _F, _I, _P, _P]),
    "biv_gemm_qkv_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "biv_rope_pack_qkv_weights": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "biv_ngram_draft": (_I, [_P, _I, _LL, _P, _I, _I, _I, _P, _P, _P]),
    "biv_lm_head_gumbel_workspace_size": (_SZ, [_I, _I, _I]),
    "biv_lm_head_gumbel": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _U64, _F, _P, _P, _SZ, _P]),
    "biv_lm_head_gumbel_accept": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _U64, _F, _P, _P, _P, _I, _I, _P, _P, _P,
                                       _SZ, _P]),
    "biv_gumbel_from_words": (_I, [_P, _LL, _P, _P]),
    "biv_verify_accept": (_I, [_P, _P, _P, _I, _I, _P, _P, _P]),
    "biv_gumbel_bucket_bounds": (_I, [_P]),
    "biv_embed": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "biv_add_rmsnorm": (_I, [_P, _P, _P, _P, _P, _I, _I, _F, _P]),
    "biv_embed_rmsnorm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P]),
    "biv_rope_qk": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _F, _P]),
    "biv_silu_mul": (_I, [_P, _P, _I, _I, _P]),
    "biv_gemm_swiglu": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "biv_swiglu_pack_weights": (_I, [_P, _P, _I, _I, _P]),
    "biv_rope_kv_write": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "biv_residual_add": (_I, [_P, _P, _P, _LL, _P]),
}


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbiv.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def lib():
    return _load()


def _check(name: str, status: int) -> None:
    if status != 0:
        raise BivError(name, status)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- status
def biv_status_string(status: int) -> str:
    return _load().biv_status_string(int(status)).decode()


def biv_version() -> int:
    return _load().biv_version()


def biv_device_error() -> int:
    bits = C.c_uint32(0)
    _check("biv_device_error", _load().biv_device_error(C.byref(bits)))
    return int(bits.value)


def biv_selftest_wait_timeout(stream=None) -> None:
    _check("biv_selftest_wait_timeout", _load().biv_selftest_wait_timeout(_stream(stream)))


# ---------------------------------------------------------------- kernels
def biv_rmsnorm(x, w, y, eps: float, stream=None) -> None:
    rows, d = x.shape
    _check("biv_rmsnorm", _load().biv_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, d, eps, _stream(stream)))


def biv_gemm_nosplitk(A, B, C_out, stream=None, bn: int | None = None) -> None:
    M, K = A.shape
    N = B.shape[0]
    dt = BIV_F32 if C_out.dtype == torch.float32 else BIV_BF16
    if bn is None:
        st = _load().biv_gemm_nosplitk(_ptr(A), _ptr(B), _ptr(C_out), dt, M, N, K, _stream(stream))
    else:
        st = _load().biv_gemm_nosplitk_bn(_ptr(A), _ptr(B), _ptr(C_out), dt, M, N, K, bn, _stream(stream))
    _check("biv_gemm_nosplitk", st)


def biv_gemm_tile_n(M: int, N: int, K: int) -> int:
    return _load().biv_gemm_tile_n(M, N, K)


def biv_decode_attn_workspace_size(W: int, Hq: int, max_len: int) -> int:
    return int(_load().biv_decode_attn_workspace_size(W, Hq, max_len))


def biv_decode_attn_fixedsplit(q, k_cache, v_cache, row_slot, row_pos, o, rows_per_group: int, workspace,
                               stream=None) -> None:
    W, Hq, hd = q.shape
    n_slots, Hkv, max_len, _ = k_cache.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("biv_decode_attn_fixedsplit", _load().biv_decode_attn_fixedsplit(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(row_slot), _ptr(row_pos), _ptr(o), W, rows_per_group,
        Hq, Hkv, hd, n_slots, max_len, KV_SPLIT, _ptr(workspace), ws_bytes, _stream(stream)))


def biv_decode_attn_fixedsplit_noalloc(q, k_cache, v_cache, row_slot, row_pos, o, rows_per_group: int,
                                       stream=None) -> None:
    """Attention without a workspace argument: the library's fixed 16 MiB
    scratch array holds the partials (for callers that cannot allocate)."""
    W, Hq, hd = q.shape
    n_slots, Hkv, max_len, _ = k_cache.shape
    _check("biv_decode_attn_fixedsplit_noalloc", _load().biv_decode_attn_fixedsplit_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(row_slot), _ptr(row_pos), _ptr(o), W, rows_per_group,
        Hq, Hkv, hd, n_slots, max_len, KV_SPLIT, _stream(stream)))


def biv_gqa_max_drafts(G: int, tile: int = ATTN_TILE) -> int:
    return _load().biv_gqa_max_drafts(G, tile)


def biv_kv_overwrite(k_cache, v_cache, k_new, v_new, row_slot, row_pos, K: int, rows_keep=None,
                     stream=None) -> None:
    """k_new / v_new: 2-D views [W, >= Hkv*hd] (row strides taken from the tensors)."""
    n_slots, Hkv, max_len, hd = k_cache.shape
    W = row_slot.shape[0]
    _check("biv_kv_overwrite", _load().biv_kv_overwrite(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_new), k_new.stride(0), _ptr(v_new), v_new.stride(0),
        _ptr(row_slot), _ptr(row_pos), _ptr(rows_keep), W, K, Hkv, hd, n_slots, max_len, _stream(stream)))


def biv_gumbel_argmax(logits, row_req, row_pos, seed: int, temperature: float, tokens, V: int | None = None,
                      stream=None) -> None:
    R, ld = logits.shape
    V = ld if V is None else V
    _check("biv_gumbel_argmax", _load().biv_gumbel_argmax(
        _ptr(logits), R, V, logits.stride(0), _ptr(row_req), _ptr(row_pos), seed & 0xFFFFFFFFFFFFFFFF,
        float(temperature), _ptr(tokens), _stream(stream)))


def biv_gumbel_argmax_workspace_size(R: int, V: int) -> int:
    return int(_load().biv_gumbel_argmax_workspace_size(R, V))


def biv_gumbel_argmax_ws(logits, row_req, row_pos, seed: int, temperature: float, tokens, workspace,
                         V: int | None = None, stream=None) -> None:
    R, ld = logits.shape
    V = ld if V is None else V
    _check("biv_gumbel_argmax_ws", _load().biv_gumbel_argmax_ws(
        _ptr(logits), R, V, logits.stride(0), _ptr(row_req), _ptr(row_pos), seed & 0xFFFFFFFFFFFFFFFF,
        float(temperature), _ptr(tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def biv_rope_pack_qkv_weights(w_qkv, w_packed, Hq: int, Hkv: int, hd: int, stream=None) -> None:
    _check("biv_rope_pack_qkv_weights", _load().biv_rope_pack_qkv_weights(
        _ptr(w_qkv), _ptr(w_packed), Hq, Hkv, hd, w_qkv.shape[1], _stream(stream)))


def biv_gemm_qkv_rope(A, B_packed, q_out, k_cache, v_cache, row_slot, row_pos, theta: float, K: int,
                      rows_keep=None, qkv_out=None, stream=None) -> None:
    W, d = A.shape
    _, Hq, hd = q_out.shape
    n_slots, Hkv, max_len, _ = k_cache.shape
    _check("biv_gemm_qkv_rope", _load().biv_gemm_qkv_rope(
        _ptr(A), _ptr(B_packed), _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(qkv_out), _ptr(row_slot),
        _ptr(row_pos), _ptr(rows_keep), W, K, d, Hq, Hkv, hd, n_slots, max_len, float(theta), _stream(stream)))


def biv_gumbel_topk(logits, row_req, row_pos, seed: int, temperature: float, out, V: int | None = None,
                    stream=None) -> None:
    R, ld = logits.shape
    V = ld if V is None else V
    k = out.shape[1]
    _check("biv_gumbel_topk", _load().biv_gumbel_topk(
        _ptr(logits), R, V, logits.stride(0), _ptr(row_req), _ptr(row_pos), seed & 0xFFFFFFFFFFFFFFFF,
        float(temperature), k, _ptr(out), _stream(stream)))


def biv_ngram_draft(hist, lengths, n_max: int, n_min: int, drafts, draft_src, stream=None) -> None:
    N, ld = hist.shape
    K = drafts.shape[1]
    _check("biv_ngram_draft", _load().biv_ngram_draft(
        _ptr(hist), N, hist.stride(0), _ptr(lengths), n_max, n_min, K, _ptr(drafts), _ptr(draft_src),
        _stream(stream)))


def biv_lm_head_gumbel_workspace_size(M: int, N: int, K: int) -> int:
    return int(_load().biv_lm_head_gumbel_workspace_size(M, N, K))


def biv_lm_head_gumbel(A, B, row_req, row_pos, seed: int, temperature: float, tokens, workspace, logits=None,
                       stream=None) -> None:
    M, K = A.shape
    N = B.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("biv_lm_head_gumbel", _load().biv_lm_head_gumbel(
        _ptr(A), _ptr(B), _ptr(logits) if logits is not None else None, M, N, K, _ptr(row_req), _ptr(row_pos),
        seed & 0xFFFFFFFFFFFFFFFF, float(temperature), _ptr(tokens), _ptr(workspace), ws_bytes, _stream(stream)))


def biv_lm_head_gumbel_accept(A, B, row_req, row_pos, seed: int, temperature: float, tokens, draft, p0,
                              n_req: int, rows_per_req: int, accept_len, new_len, workspace, logits=None,
                              stream=None) -> None:
    M, K = A.shape
    N = B.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("biv_lm_head_gumbel_accept", _load().biv_lm_head_gumbel_accept(
        _ptr(A), _ptr(B), _ptr(logits) if logits is not None else None, M, N, K, _ptr(row_req), _ptr(row_pos),
        seed & 0xFFFFFFFFFFFFFFFF, float(temperature), _ptr(tokens), _ptr(draft), _ptr(p0), n_req, rows_per_req,
        _ptr(accept_len), _ptr(new_len), _ptr(workspace), ws_bytes, _stream(stream)))


def biv_gumbel_noise(seed: int, row_req, row_pos, g, stream=None) -> None:
    R, V = g.shape
    _check("biv_gumbel_noise", _load().biv_gumbel_noise(
        seed & 0xFFFFFFFFFFFFFFFF, _ptr(row_req), _ptr(row_pos), R, V, _ptr(g), _stream(stream)))


def biv_gumbel_from_words(words, g, stream=None) -> None:
    _check("biv_gumbel_from_words", _load().biv_gumbel_from_words(
        _ptr(words), words.numel(), _ptr(g), _stream(stream)))


def biv_gumbel_bucket_bounds():
    import numpy as np
    out = np.empty(256, np.float32)
    _check("biv_gumbel_bucket_bounds", _load().biv_gumbel_bucket_bounds(out.ctypes.data_as(C.c_void_p)))
    return out


def biv_verify_accept(target, draft, p0, N: int, K: int, accept_len, new_len, stream=None) -> None:
    _check("biv_verify_accept", _load().biv_verify_accept(
        _ptr(target), _ptr(draft), _ptr(p0), N, K, _ptr(accept_len), _ptr(new_len), _stream(stream)))


def biv_add_rmsnorm(x, r, w, x_out, y, eps: float, stream=None) -> None:
    rows, d = x.shape
    _check("biv_add_rmsnorm", _load().biv_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), _ptr(x_out), _ptr(y), rows, d,
                                                      eps, _stream(stream)))


def biv_embed_rmsnorm(table, tokens, w, x_out, y, eps: float, stream=None) -> None:
    vocab, d = table.shape
    _check("biv_embed_rmsnorm", _load().biv_embed_rmsnorm(_ptr(table), _ptr(tokens), _ptr(w), _ptr(x_out), _ptr(y),
                                                          tokens.shape[0], d, vocab, eps, _stream(stream)))


def biv_embed(table, tokens, out, stream=None) -> None:
    vocab, d = table.shape
    _check("biv_embed", _load().biv_embed(_ptr(table), _ptr(tokens), _ptr(out), tokens.shape[0], d, vocab,
                                          _stream(stream)))


def biv_rope_qk(qkv, q_out, k_out, row_pos, Hq: int, Hkv: int, hd: int, theta: float, stream=None) -> None:
    W = qkv.shape[0]
    _check("biv_rope_qk", _load().biv_rope_qk(_ptr(qkv), _ptr(q_out), _ptr(k_out), _ptr(row_pos), W, Hq, Hkv, hd,
                                              float(theta), _stream(stream)))


def biv_silu_mul(gu, out, stream=None) -> None:
    rows, two_f = gu.shape
    _check("biv_silu_mul", _load().biv_silu_mul(_ptr(gu), _ptr(out), rows, two_f // 2, _stream(stream)))


def biv_gemm_swiglu(A, B_packed, act, stream=None) -> None:
    M, K = A.shape
    F = act.shape[1]
    _check("biv_gemm_swiglu", _load().biv_gemm_swiglu(_ptr(A), _ptr(B_packed), _ptr(act), M, F, K,
                                                      _stream(stream)))


def biv_swiglu_pack_weights(w_gu, w_packed, stream=None) -> None:
    two_f, K = w_gu.shape
    _check("biv_swiglu_pack_weights", _load().biv_swiglu_pack_weights(_ptr(w_gu), _ptr(w_packed), two_f // 2, K,
                                                                      _stream(stream)))


def biv_rope_kv_write(qkv, q_out, k_cache, v_cache, row_slot, row_pos, Hq: int, theta: float, K: int,
                      rows_keep=None, stream=None) -> None:
    n_slots, Hkv, max_len, hd = k_cache.shape
    W = qkv.shape[0]
    _check("biv_rope_kv_write", _load().biv_rope_kv_write(
        _ptr(qkv), _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(row_slot), _ptr(row_pos), _ptr(rows_keep),
        W, K, Hq, Hkv, hd, n_slots, max_len, float(theta), _stream(stream)))


def biv_residual_add(x, y, out, stream=None) -> None:
    _check("biv_residual_add", _load().biv_residual_add(_ptr(x), _ptr(y), _ptr(out), x.numel(), _stream(stream)))
