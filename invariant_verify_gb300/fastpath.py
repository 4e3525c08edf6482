"""The batch-variant fast path as a drafter, and the Decode-Verify-Rollback loop.

Decode-Verify-Rollback (tgstat @ashnskt post 392, paragraph 3): a fast,
batch-variant engine decodes ahead at whatever batch it has; a fixed-shape
batch-invariant verifier recomputes the window and is the ground truth; the
output rolls back to the last token the verifier agrees with, and the fast
path's KV rows are overwritten with the verifier's values.  With coupled
Gumbel selection (AIexTime post 185) the fast path's tokens only decide how
many verified tokens a step commits, never which ones.

The fast path is ordinary PyTorch on cuBLAS (free to split K and to change
its reduction order with the batch size) and scaled-dot-product attention
over its own KV cache; only its token selection is the library's Gumbel-max
with the verifier's noise.  It is a drafter, not the verified path.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.nn.functional as F

from . import abi as B
from .verifier import DecoderVerifier, make_window


def _rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps) * w.float()).to(torch.bfloat16)


def _rope(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half RoPE of x [n, H, hd] at positions pos [n] (fp32 math)."""
    hd = x.shape[-1]
    inv = theta ** (-torch.arange(0, hd // 2, device=x.device, dtype=torch.float32) * 2.0 / hd)
    ang = pos.float()[:, None] * inv[None, :]
    cos, sin = ang.cos()[:, None, :], ang.sin()[:, None, :]
    xf = x.float()
    a, b = xf[..., : hd // 2], xf[..., hd // 2:]
    return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1).to(torch.bfloat16)


class FastPathDecoder:
    """Batch-variant decoder over its own KV cache (the drafter of the DVR loop)."""

    def __init__(self, cfg, weights: dict, caches: list, seed: int):
        self.cfg, self.seed = cfg, seed
        self.w = weights
        self.kc = [k.clone() for k, _ in caches]
        self.vc = [v.clone() for _, v in caches]

    @torch.no_grad()
    def step(self, tokens: torch.Tensor, pos: torch.Tensor, slots: torch.Tensor, req: torch.Tensor) -> torch.Tensor:
        """One decode step for a batch of requests: input token at position
        pos (int32 [n], device) -> the selected next token (int32 [n])."""
        c, w = self.cfg, self.w
        n = tokens.shape[0]
        Hq, Hkv, hd = c.Hq, c.Hkv, c.hd
        x = w["embed"][tokens.long()]
        posl, sl = pos.long(), slots.long()
        lmax = int(pos.max().item()) + 1
        keep = torch.arange(lmax, device=x.device)[None, :] <= posl[:, None]        # [n, lmax]
        mask = torch.zeros(n, 1, 1, lmax, device=x.device, dtype=torch.bfloat16)
        mask.masked_fill_(~keep[:, None, None, :], float("-inf"))
        for l in range(c.layers):
            h = _rmsnorm(x, w[f"l{l}.attn_norm"], c.eps)
            qkv = h @ w[f"l{l}.wqkv"].t()
            q = _rope(qkv[:, : Hq * hd].view(n, Hq, hd), pos, c.rope_theta)
            k = _rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].view(n, Hkv, hd), pos, c.rope_theta)
            v = qkv[:, (Hq + Hkv) * hd:].view(n, Hkv, hd)
            self.kc[l][sl, :, posl] = k
            self.vc[l][sl, :, posl] = v
            kk = self.kc[l][sl, :, :lmax]                                             # [n, Hkv, lmax, hd]
            vv = self.vc[l][sl, :, :lmax]
            o = F.scaled_dot_product_attention(q[:, :, None, :], kk, vv, attn_mask=mask, enable_gqa=True)
            x = x + o.reshape(n, Hq * hd) @ w[f"l{l}.wo"].t()
            h = _rmsnorm(x, w[f"l{l}.ffn_norm"], c.eps)
            gu = h @ w[f"l{l}.wgu"].t()
            g, u = gu[:, : c.ffn], gu[:, c.ffn:]
            x = x + (F.silu(g.float()) * u.float()).to(torch.bfloat16) @ w[f"l{l}.wdown"].t()
        h = _rmsnorm(x, w["final_norm"], c.eps)
        logits = (h @ w["lm_head"].t()).float()
        tok = torch.empty(n, dtype=torch.int32, device=x.device)
        B.biv_gumbel_argmax(logits, req, pos, self.seed, c.temperature, tok)
        return tok

    def overwrite(self, ver: DecoderVerifier, slots: torch.Tensor, p0: torch.Tensor, n_rows: torch.Tensor) -> None:
        """Copy the verifier's K/V rows [p0, p0 + n_rows) of each slot into the fast cache."""
        for r in range(slots.shape[0]):
            s, a, b = int(slots[r]), int(p0[r]), int(p0[r] + n_rows[r])
            for l in range(self.cfg.layers):
                self.kc[l][s, :, a:b] = ver.kc[l][s, :, a:b]
                self.vc[l][s, :, a:b] = ver.vc[l][s, :, a:b]


@dataclass
class DvrStats:
    rounds: int = 0
    drafted: int = 0          # draft tokens proposed
    accepted: int = 0         # draft tokens the verifier agreed with
    committed: int = 0        # tokens committed (accepted + one verifier token per round)

    @property
    def divergence_rate(self) -> float:
        return 1.0 - self.accepted / max(1, self.drafted)


@torch.no_grad()
def dvr_generate(ver: DecoderVerifier, fast: FastPathDecoder | None, last_tokens: torch.Tensor, p0: torch.Tensor,
                 req: torch.Tensor, n_tokens: int) -> tuple[list[torch.Tensor], DvrStats]:
    """Generate n_tokens per request with Decode-Verify-Rollback.

    ver: verifier with W = N * K rows, K = ver.rpg, request r in cache slot r;
    last_tokens, p0, req: int32 [N] (host) -- the last committed token, its
    position, the stable request id.  fast = None verifies without drafts
    (every round commits exactly one token).  Returns the committed tokens of
    each request and the loop's statistics."""
    N, K = last_tokens.shape[0], ver.rpg
    dev = ver.target.device
    slots = torch.arange(N, dtype=torch.int32)
    last, pos = last_tokens.clone().to(torch.int32), p0.clone().to(torch.int32)
    out = [[] for _ in range(N)]
    st = DvrStats()
    while min(len(o) for o in out) < n_tokens:
        drafts = torch.zeros(N, K, dtype=torch.int32)
        if fast is not None and K > 1:
            # the fast path decodes K tokens ahead at batch N (its own batch shape)
            t, p = last.to(dev), pos.to(dev)
            for j in range(K):
                nxt = fast.step(t, p, slots.to(dev), req.to(dev))
                drafts[:, j] = nxt.cpu()
                t, p = nxt, p + 1
        tokens = torch.cat([last[:, None], drafts[:, :-1]], dim=1)
        win = make_window(N, K, tokens.reshape(-1), pos, req, drafts.reshape(-1), device=dev)
        ver.step(win)
        L = ver.accept_len.cpu()
        tgt = ver.target.view(N, K).cpu()
        if fast is not None:
            fast.overwrite(ver, slots, pos, L)           # the fast cache takes the verified rows
        st.rounds += 1
        if fast is not None and K > 1:
            st.drafted += N * K
            st.accepted += int(sum(int(L[r]) - (0 if int(L[r]) == K and bool((tgt[r] == drafts[r]).all()) else 1)
                                   for r in range(N)))
        for r in range(N):
            n = int(L[r])
            out[r].extend(tgt[r, :n].tolist())
            st.committed += n
            last[r] = tgt[r, n - 1]
            pos[r] += n
    return [torch.tensor(o[:n_tokens], dtype=torch.int32) for o in out], st
