"""Seeded synthetic inputs for the verification step.

This module only draws random numbers and arranges them into the shapes of
the workloads; it holds none of the method's arithmetic (no normalisation,
no products, no noise, no selection).  Both the CUDA path and the CPU
oracle read their inputs from here, so the two sides always see the same
bytes.

All tensors are CPU torch tensors (bf16 weights/activations, fp32 logits,
int32 ids).  Every generator takes an integer seed and is deterministic.

Workloads (sizes as the verification-step pages describe them):

* ``TINY``      -- RMSNorm(d=256) -> LM head [W x 256]x[256 x 2048] -> select,
                   N=4 requests x K=4 tokens.
* ``DECODER2``  -- random-init 2-layer decoder verifier, d=1024, 8 query /
                   2 KV heads of 128, SwiGLU 2816, vocab 32000, N=8 x K=8.
* ``LLAMA8B``   -- one Llama-3-8B-shaped layer + LM head (d=4096, 32/8 heads,
                   FFN 14336, vocab 128256), decode rows M in {1..256}, KV 4096.
* ``SWEEP``     -- the LLAMA8B shapes verified at N in {8,32,64} x K in {4,8,16}
                   with lognormal context lengths.
* ``SELECT``    -- bandwidth-bound selection over fp32 logits
                   [512 x 8 rows x 152064], T=0.7.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = [
    "DecoderConfig", "TINY", "DECODER2", "LLAMA8B", "SWEEP", "SELECT",
    "generator", "bf16_normal", "decoder_weights", "context_lengths",
    "kv_cache", "request_window", "draft_errors", "apply_draft_errors",
    "select_logits", "tiny_inputs",
]

PHILOX_SEED = 0x1234_5678_9ABC_DEF0


@dataclass(frozen=True)
class DecoderConfig:
    name: str
    layers: int
    d: int
    Hq: int
    Hkv: int
    hd: int
    ffn: int
    vocab: int
    eps: float = 1e-6
    w_std: float = 0.02
    rope_theta: float = 10000.0
    kv_split: int = 256
    N: int = 8
    K: int = 8
    temperature: float = 0.7
    draft_err: float = 0.3
    ctx: str = "uniform"            # "uniform" | "lognormal" | "fixed"
    ctx_lo: int = 128
    ctx_hi: int = 2048
    ctx_median: float = 1024.0
    ctx_sigma: float = 1.0
    seed: int = 2

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def W(self) -> int:
        return self.N * self.K

    @property
    def qkv_n(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.hd


@dataclass(frozen=True)
class TinyConfig:
    name: str = "tiny: rmsnorm d256 + lm-head 2048, N4xK4"
    d: int = 256
    vocab: int = 2048
    N: int = 4
    K: int = 4
    temperature: float = 1.0
    w_std: float = 1.0 / 16.0       # N(0, 1/256)
    h_std: float = 1.0
    draft_err: float = 0.25
    eps: float = 1e-6
    seed: int = 1
    invariance_W: tuple = (1, 2, 4, 8, 16)


@dataclass(frozen=True)
class SelectConfig:
    name: str = "select: fp32 logits 4096x152064, T0.7"
    requests: int = 512
    K: int = 8
    vocab: int = 152064
    temperature: float = 0.7
    base_std: float = 3.0
    peak: float = 10.0
    peaked_frac: float = 0.9
    tie_gap: float = 1e-3
    draft_err: float = 0.2
    seed: int = 5

    @property
    def R(self) -> int:
        return self.requests * self.K


TINY = TinyConfig()
DECODER2 = DecoderConfig(name="decoder-2L d1024 8q/2kv ffn2816 v32000, N8xK8",
                         layers=2, d=1024, Hq=8, Hkv=2, hd=128, ffn=2816,
                         vocab=32000, rope_theta=10000.0, N=8, K=8,
                         temperature=0.7, draft_err=0.3, ctx="uniform",
                         ctx_lo=128, ctx_hi=2048, seed=2)
LLAMA8B = DecoderConfig(name="llama3-8b-shaped layer + lm-head, KV 4096",
                        layers=1, d=4096, Hq=32, Hkv=8, hd=128, ffn=14336,
                        vocab=128256, rope_theta=500000.0, N=256, K=1,
                        temperature=0.7, draft_err=0.2, ctx="fixed",
                        ctx_lo=4096, ctx_hi=4096, seed=3)
SWEEP = DecoderConfig(name="llama3-8b-shaped verifier sweep, lognormal ctx",
                      layers=1, d=4096, Hq=32, Hkv=8, hd=128, ffn=14336,
                      vocab=128256, rope_theta=500000.0, N=64, K=16,
                      temperature=0.7, draft_err=0.2, ctx="lognormal",
                      ctx_lo=256, ctx_hi=8192, ctx_median=1024.0,
                      ctx_sigma=1.0, seed=4)
SELECT = SelectConfig()


def generator(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def bf16_normal(shape, std: float, gen: torch.Generator) -> torch.Tensor:
    """N(0, std^2) samples rounded to bf16 (round-to-nearest-even by torch)."""
    return (torch.randn(*shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def bf16_normal_device(shape, std: float, seed: int, device="cuda") -> torch.Tensor:
    """N(0, std^2) bf16 samples drawn on the device with a seeded generator
    (for multi-GB inputs; the stream differs from the CPU generator's)."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def decoder_weights_device(cfg: DecoderConfig, seed: int | None = None, device="cuda") -> dict:
    """Like decoder_weights, drawn on the device (same layout, other stream)."""
    s0 = cfg.seed if seed is None else seed
    w = {"embed": bf16_normal_device((cfg.vocab, cfg.d), cfg.w_std, s0 * 1000 + 1, device)}
    for l in range(cfg.layers):
        b = s0 * 1000 + 10 * (l + 1)
        w[f"l{l}.attn_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16, device=device)
        w[f"l{l}.wqkv"] = bf16_normal_device((cfg.qkv_n, cfg.d), cfg.w_std, b + 1, device)
        w[f"l{l}.wo"] = bf16_normal_device((cfg.d, cfg.Hq * cfg.hd), cfg.w_std, b + 2, device)
        w[f"l{l}.ffn_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16, device=device)
        w[f"l{l}.wgu"] = bf16_normal_device((2 * cfg.ffn, cfg.d), cfg.w_std, b + 3, device)
        w[f"l{l}.wdown"] = bf16_normal_device((cfg.d, cfg.ffn), cfg.w_std, b + 4, device)
    w["final_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16, device=device)
    w["lm_head"] = bf16_normal_device((cfg.vocab, cfg.d), cfg.w_std, s0 * 1000 + 2, device)
    return w


def kv_cache_device(n_slots: int, Hkv: int, max_len: int, hd: int, ctx: torch.Tensor, seed: int,
                    layers: int = 1, device="cuda") -> list:
    """Like kv_cache, drawn on the device: N(0,1) below ctx[slot], zero above."""
    out = []
    pos = torch.arange(max_len, device=device)
    keep = (pos[None, :] < ctx.to(device)[:, None])[:, None, :, None]
    for l in range(layers):
        pair = []
        for kv in range(2):
            c = bf16_normal_device((n_slots, Hkv, max_len, hd), 1.0, seed * 100 + 2 * l + kv, device)
            pair.append(torch.where(keep, c, torch.zeros((), dtype=c.dtype, device=device)).contiguous())
        out.append(tuple(pair))
    return out


def decoder_weights(cfg: DecoderConfig, seed: int | None = None) -> dict:
    """Random-init decoder verifier weights, nn.Linear layout [out, in].

    Norm gains are ones: the workloads state N(0, 0.02) for weights but say
    nothing about gains, and gains drawn from N(0, 0.02) would scale the
    signal to nothing.  The gate/up projection is one [2F, d] matrix with
    the F gate rows first.
    """
    g = generator(cfg.seed if seed is None else seed)
    w = {"embed": bf16_normal((cfg.vocab, cfg.d), cfg.w_std, g)}
    for l in range(cfg.layers):
        w[f"l{l}.attn_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16)
        w[f"l{l}.wqkv"] = bf16_normal((cfg.qkv_n, cfg.d), cfg.w_std, g)
        w[f"l{l}.wo"] = bf16_normal((cfg.d, cfg.Hq * cfg.hd), cfg.w_std, g)
        w[f"l{l}.ffn_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16)
        w[f"l{l}.wgu"] = bf16_normal((2 * cfg.ffn, cfg.d), cfg.w_std, g)
        w[f"l{l}.wdown"] = bf16_normal((cfg.d, cfg.ffn), cfg.w_std, g)
    w["final_norm"] = torch.ones(cfg.d, dtype=torch.bfloat16)
    w["lm_head"] = bf16_normal((cfg.vocab, cfg.d), cfg.w_std, g)
    return w


def context_lengths(cfg: DecoderConfig, n: int, seed: int) -> torch.Tensor:
    """Per-request cached context lengths (int32 [n])."""
    g = generator(seed)
    if cfg.ctx == "uniform":
        return torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    if cfg.ctx == "lognormal":
        z = torch.randn(n, generator=g, dtype=torch.float64)
        c = torch.round(cfg.ctx_median * torch.exp(cfg.ctx_sigma * z))
        return c.clamp(cfg.ctx_lo, cfg.ctx_hi).to(torch.int32)
    return torch.full((n,), cfg.ctx_lo, dtype=torch.int32)


def kv_cache(n_slots: int, Hkv: int, max_len: int, hd: int, ctx: torch.Tensor,
             seed: int, layers: int = 1) -> list:
    """Per-layer (K, V) caches, bf16 [n_slots, Hkv, max_len, hd].

    Positions below ctx[slot] hold N(0,1) values; the rest are zero.
    """
    g = generator(seed)
    out = []
    for _ in range(layers):
        pair = []
        for _kv in range(2):
            c = torch.zeros(n_slots, Hkv, max_len, hd, dtype=torch.bfloat16)
            for s in range(n_slots):
                n = int(ctx[s])
                c[s, :, :n, :] = bf16_normal((Hkv, n, hd), 1.0, g)
            pair.append(c)
        out.append(tuple(pair))
    return out


def request_window(N: int, K: int, p0: torch.Tensor, req_ids: torch.Tensor | None = None):
    """Row metadata of a W = N*K verify window, request-major.

    Row r*K + j belongs to request r, sits in cache slot r and at absolute
    position p0[r] + j.  Returns (row_slot, row_req, row_pos) int32 [W].
    """
    if req_ids is None:
        req_ids = torch.arange(N, dtype=torch.int32)
    r = torch.arange(N, dtype=torch.int32).repeat_interleave(K)
    j = torch.arange(K, dtype=torch.int32).repeat(N)
    return r.clone(), req_ids.to(torch.int32)[r.long()].clone(), (p0.to(torch.int32)[r.long()] + j).to(torch.int32)


def draft_errors(shape, rate: float, vocab: int, seed: int):
    """Where a drafter errs (bool mask) and the uniform ids it then proposes."""
    g = generator(seed)
    mask = torch.rand(*shape, generator=g) < rate
    ids = torch.randint(0, vocab, shape, generator=g, dtype=torch.int64).to(torch.int32)
    return mask, ids


def apply_draft_errors(target: torch.Tensor, mask: torch.Tensor, ids: torch.Tensor) -> torch.Tensor:
    return torch.where(mask, ids, target).to(torch.int32)


def select_logits(cfg: SelectConfig = SELECT, rows: int | None = None, seed: int | None = None,
                  exact_ties: bool = False) -> tuple:
    """fp32 logits for the selection workload and the kind of each row.

    Peaked rows (``kind == 0``): N(0, base_std^2) with one random index set
    to the row maximum + peak.  Near-tie rows (``kind == 1``): N(0, base_std^2)
    with a second index set to the row maximum minus delta, delta ~ U(0, gap);
    with ``exact_ties`` delta is 0 so the lowest-index rule decides.
    """
    R = cfg.R if rows is None else rows
    V = cfg.vocab
    g = generator(cfg.seed if seed is None else seed)
    x = torch.randn(R, V, generator=g, dtype=torch.float32) * cfg.base_std
    kind = (torch.rand(R, generator=g) >= cfg.peaked_frac).to(torch.int32)
    i1 = torch.randint(0, V, (R,), generator=g)
    i2 = torch.randint(0, V, (R,), generator=g)
    i2 = torch.where(i2 == i1, (i1 + 1) % V, i2)
    delta = torch.rand(R, generator=g, dtype=torch.float32) * cfg.tie_gap
    if exact_ties:
        delta.zero_()
    rmax = x.max(dim=1).values
    ar = torch.arange(R)
    peaked = kind == 0
    x[ar[peaked], i1[peaked]] = rmax[peaked] + cfg.peak
    tie = ~peaked
    x[ar[tie], i1[tie]] = rmax[tie]
    x[ar[tie], i2[tie]] = rmax[tie] - delta[tie]
    return x, kind


def select_logits_device(cfg: SelectConfig = SELECT, seed: int | None = None, device="cuda") -> torch.Tensor:
    """select_logits' recipe drawn on the device (the full 2.49 GB workload)."""
    R, V = cfg.R, cfg.vocab
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed if seed is None else seed)
    x = torch.randn(R, V, generator=g, device=device, dtype=torch.float32) * cfg.base_std
    kind = (torch.rand(R, generator=g, device=device) >= cfg.peaked_frac)
    i1 = torch.randint(0, V, (R,), generator=g, device=device)
    i2 = torch.randint(0, V, (R,), generator=g, device=device)
    i2 = torch.where(i2 == i1, (i1 + 1) % V, i2)
    delta = torch.rand(R, generator=g, device=device, dtype=torch.float32) * cfg.tie_gap
    rmax = x.max(dim=1).values
    ar = torch.arange(R, device=device)
    x[ar, i1] = torch.where(kind, rmax, rmax + cfg.peak)
    x[ar[kind], i2[kind]] = (rmax - delta)[kind]
    return x


def tiny_inputs(cfg: TinyConfig = TINY, seed: int | None = None) -> dict:
    g = generator(cfg.seed if seed is None else seed)
    W = cfg.N * cfg.K
    h = bf16_normal((W, cfg.d), cfg.h_std, g)
    lm = bf16_normal((cfg.vocab, cfg.d), cfg.w_std, g)
    p0 = torch.randint(16, 4000, (cfg.N,), generator=g, dtype=torch.int64).to(torch.int32)
    req = torch.randint(0, 2**31 - 1, (cfg.N,), generator=g, dtype=torch.int64).to(torch.int32)
    return dict(h=h, lm_head=lm, gain=torch.ones(cfg.d, dtype=torch.bfloat16), p0=p0, req_ids=req)
