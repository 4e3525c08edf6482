"""Oracle composition of one verify forward and of the Decode-Verify-Rollback loop.

Test infrastructure only (see the package docstring).  Each step calls the
plain C++ primitives of ``oracle.cpp``; nothing is fused or reordered.

The layer is the standard pre-norm Llama decoder -- a reading, since the
pages describe the verifier only as "a forward pass at a fixed batch size"
([DVR] para 3):

    x = embed[token]
    per layer:  h = rmsnorm(x); qkv = h W_qkv^T; q,k = rope(q,k, pos);
                write k,v at the rows' positions; o = attn(q, cache);
                x = x + o W_o^T; h = rmsnorm(x); a = silu(gate) * up;
                x = x + a W_down^T
    logits = rmsnorm(x) W_lm^T

``storage="bf16"`` rounds every stored activation to bf16 at the points
where a bf16 verifier stores them (GEMM outputs, norm outputs, RoPE output,
residual stream, attention output); logits stay fp32.  ``storage="f64"``
keeps every intermediate in fp64.  The KV cache is bf16 in both modes.
``storage="bf16_random"`` stores at the same points but rounds each element
to one of its two bracketing bf16 values at random (``rng``), the window's
K/V rows included: the drift envelope of implementations that round within
one ulp at every storage point.
"""
from __future__ import annotations

import numpy as np

from . import (_f64, _np, attention, from_bf16, gemm, gumbel_argmax, kv_overwrite, rmsnorm,
               rope, round_bf16, round_bf16_random, silu_mul, to_bf16, verify_accept)


class OracleDecoder:
    def __init__(self, cfg, weights: dict, caches: list, n_slots: int, max_len: int):
        """weights: name -> bf16 tensor/uint16 array; caches: per layer (K, V) bf16."""
        self.cfg = cfg
        self.w = {k: _np(v) for k, v in weights.items()}
        self.gain = {k: from_bf16(v) for k, v in self.w.items() if k.endswith("norm")}
        self.caches = [(np.ascontiguousarray(_np(k)).copy(), np.ascontiguousarray(_np(v)).copy())
                       for k, v in caches]
        self.n_slots, self.max_len = n_slots, max_len

    def forward(self, tokens, row_slot, row_pos, storage: str = "bf16", rng=None) -> dict:
        cfg = self.cfg
        if storage == "bf16_random":
            R = lambda a: round_bf16_random(a, rng)
            KV = lambda a: to_bf16(round_bf16_random(a, rng))
        else:
            R = round_bf16 if storage == "bf16" else (lambda a: a)
            KV = to_bf16
        tok = np.ascontiguousarray(_np(tokens), np.int64)
        rs = np.ascontiguousarray(_np(row_slot), np.int32)
        rp = np.ascontiguousarray(_np(row_pos), np.int32)
        W = tok.size
        x = from_bf16(self.w["embed"][tok])
        Hq, Hkv, hd = cfg.Hq, cfg.Hkv, cfg.hd
        for l in range(cfg.layers):
            h = R(rmsnorm(x, self.gain[f"l{l}.attn_norm"], cfg.eps))
            qkv = R(gemm(h, self.w[f"l{l}.wqkv"]))
            q = qkv[:, : Hq * hd].reshape(W, Hq, hd)
            k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(W, Hkv, hd)
            v = qkv[:, (Hq + Hkv) * hd:].reshape(W, Hkv, hd)
            q = R(rope(q, rp, cfg.rope_theta))
            k = rope(k, rp, cfg.rope_theta)
            kc, vc = self.caches[l]
            kv_overwrite(kc, vc, KV(k), KV(v), rs, rp)
            o = R(attention(q, kc, vc, rs, rp))
            x = R(x + R(gemm(o.reshape(W, Hq * hd), self.w[f"l{l}.wo"])))
            h = R(rmsnorm(x, self.gain[f"l{l}.ffn_norm"], cfg.eps))
            gu = R(gemm(h, self.w[f"l{l}.wgu"]))
            a = R(silu_mul(gu))
            x = R(x + R(gemm(a, self.w[f"l{l}.wdown"])))
        hf = R(rmsnorm(x, self.gain["final_norm"], cfg.eps))
        logits = gemm(hf, self.w["lm_head"])
        if storage != "f64":
            logits = logits.astype(np.float32).astype(np.float64)
        return {"hidden": hf, "logits": logits}

    def verify(self, tokens, row_slot, row_req, row_pos, draft, p0, N, K, seed, temperature,
               storage: str = "bf16") -> dict:
        out = self.forward(tokens, row_slot, row_pos, storage)
        tgt = gumbel_argmax(out["logits"].astype(np.float32), row_req, row_pos, seed, temperature)
        L, new_len = verify_accept(tgt, draft, p0, N, K)
        out.update(target=tgt, accept_len=L, new_len=new_len)
        return out


def dvr_decode(model: OracleDecoder, first_tokens, p0, req_ids, n_tokens: int, K: int, drafter,
               seed: int, temperature: float, storage: str = "bf16") -> list:
    """Decode-Verify-Rollback until every request has ``n_tokens`` new tokens.

    ``drafter(r, history, K)`` proposes K draft tokens d_1..d_K for request r
    (history = committed tokens so far).  Each round verifies K rows per
    request: row j takes the last committed token (j = 0) or d_j, sits at
    position p0 + j, and its selected token y_{j+1} is compared with d_{j+1}.
    y_1..y_L are committed, p0 advances to p0 + L (rollback of the rest).
    Returns the committed streams, one list per request.
    """
    N = len(first_tokens)
    last = [int(t) for t in first_tokens]
    pos = [int(p) for p in p0]
    streams = [[] for _ in range(N)]
    while min(len(s) for s in streams) < n_tokens:
        drafts = np.array([drafter(r, streams[r], K) for r in range(N)], np.int32).reshape(N, K)
        tokens = np.empty((N, K), np.int32)
        tokens[:, 0] = last
        tokens[:, 1:] = drafts[:, :-1]
        row_slot = np.repeat(np.arange(N, dtype=np.int32), K)
        row_req = np.repeat(np.asarray(req_ids, np.int64), K)
        row_pos = (np.repeat(np.asarray(pos, np.int32), K) + np.tile(np.arange(K, dtype=np.int32), N))
        out = model.verify(tokens.reshape(-1), row_slot, row_req, row_pos, drafts.reshape(-1),
                           np.asarray(pos, np.int32), N, K, seed, temperature, storage)
        tgt = out["target"].reshape(N, K)
        for r in range(N):
            L = int(out["accept_len"][r])
            streams[r].extend(int(t) for t in tgt[r, :L])
            last[r] = int(tgt[r, L - 1])
            pos[r] += L
    return [s[:n_tokens] for s in streams]
