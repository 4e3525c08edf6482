"""Composition of one batch-invariant verify step out of libbiv calls.

Decode-Verify-Rollback ([DVR] paras 3-4, tgstat @ashnskt post 392): the
verifier runs one fixed-shape forward over W = N requests x K tokens, writes
its own K/V for the window rows into the cache (overwriting whatever the
fast path left there), selects one token per row with shared Gumbel noise,
and compares the selections with the drafts ([COUPLING], AIexTime post 185).

Every arithmetic step runs in libbiv's CUDA kernels; this module only owns
device buffers and issues the C-ABI calls in order on one stream.  The layer
is the standard pre-norm Llama decoder (a reading: the pages do not describe
the verifier model).

Row layout of a window (request-major): row r*K + j holds the last committed
token (j = 0) or draft d_j, sits in cache slot row_slot and at absolute
position p0[r] + j; its selected token y_{j+1} is compared with
draft[r*K + j] = d_{j+1}.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import abi as B


@dataclass
class Window:
    """Device-resident row metadata and drafts of one verify window."""
    tokens: torch.Tensor     # int32 [W] input token per row
    row_slot: torch.Tensor   # int32 [W]
    row_req: torch.Tensor    # int32 [W] (stable request id, used as uint32)
    row_pos: torch.Tensor    # int32 [W]
    draft: torch.Tensor      # int32 [W] draft each row's selection must match
    p0: torch.Tensor         # int32 [N]


class DecoderVerifier:
    """Device-resident decoder verifier for windows of exactly W rows.

    ``fused_select``: the LM-head GEMM selects each row's token in its
    epilogue (biv_lm_head_gumbel), bit-identical to the LM head followed by
    biv_gumbel_argmax; ``keep_logits`` then decides whether the fp32 logits
    are also stored (they always are without fusion)."""

    def __init__(self, cfg, weights: dict, caches: list, n_slots: int, max_len: int, W: int,
                 rows_per_group: int, device="cuda", seed: int = 0x1234_5678_9ABC_DEF0,
                 fused_select: bool = True, keep_logits: bool = True):
        self.cfg, self.W, self.rpg = cfg, W, rows_per_group
        self.fused_select = fused_select
        self.keep_logits = keep_logits or not fused_select
        self.n_slots, self.max_len, self.seed = n_slots, max_len, seed
        dev = torch.device(device)
        self.w = {k: v.to(dev).contiguous() for k, v in weights.items()}
        # gate/up weights rearranged once for the SwiGLU-epilogue GEMM
        for l in range(cfg.layers):
            wgu = self.w[f"l{l}.wgu"]
            packed = torch.empty_like(wgu)
            B.biv_swiglu_pack_weights(wgu, packed)
            self.w[f"l{l}.wgu_packed"] = packed
            # QKV rows rearranged once for the RoPE/KV-write epilogue
            wqkv = self.w[f"l{l}.wqkv"]
            rpk = torch.empty_like(wqkv)
            B.biv_rope_pack_qkv_weights(wqkv, rpk, cfg.Hq, cfg.Hkv, cfg.hd)
            self.w[f"l{l}.wqkv_rope"] = rpk
        self.kc = [k.to(dev).contiguous() for k, _ in caches]
        self.vc = [v.to(dev).contiguous() for _, v in caches]
        d, Hq, Hkv, hd, F = cfg.d, cfg.Hq, cfg.Hkv, cfg.hd, cfg.ffn
        bf = dict(device=dev, dtype=torch.bfloat16)
        self.x = torch.empty(W, d, **bf)
        self.h = torch.empty(W, d, **bf)
        self.qkv = torch.empty(W, cfg.qkv_n, **bf)
        self.q = torch.empty(W, Hq, hd, **bf)
        self.o = torch.empty(W, Hq, hd, **bf)
        self.proj = torch.empty(W, d, **bf)
        self.act = torch.empty(W, F, **bf)
        self.hidden = torch.empty(W, d, **bf)
        self.logits = torch.empty(W, cfg.vocab, device=dev, dtype=torch.float32) if self.keep_logits else None
        if fused_select:
            n = B.biv_lm_head_gumbel_workspace_size(W, cfg.vocab, d)
            self.select_ws = torch.empty(max(n, 16), device=dev, dtype=torch.uint8)
        N = (W + rows_per_group - 1) // rows_per_group
        # the step's results, [accept_len N | new_len N | target W], in one
        # buffer so that one copy reads them back
        self.results = torch.empty(2 * N + W, device=dev, dtype=torch.int32)
        self.accept_len = self.results[:N]
        self.new_len = self.results[N:2 * N]
        self.target = self.results[2 * N:]
        ws = B.biv_decode_attn_workspace_size(W, Hq, max_len)
        self.workspace = torch.empty(max(ws, 16), device=dev, dtype=torch.uint8)
        # embed+norm; per layer QKV+RoPE, attention (two), Wo, add+norm,
        # gate/up+SwiGLU, down, add+norm; then the LM head with the selection
        # and one winners+accept kernel, or the LM head, selection and accept
        self.launches_per_step = (3 if fused_select else 4) + cfg.layers * 8

    # -------------------------------------------------------------- stages
    def forward(self, win: Window, trace: dict | None = None, mark=None) -> None:
        """Hidden state of every window row (cache rows written).

        ``trace``, if given, receives a copy of every intermediate (for
        stage-by-stage parity tests); it adds device copies, so it is not for
        the timed path.  ``mark``, if given, is called with a stage name after
        each library call (a benchmark records a timing event there).
        """
        c, w = self.cfg, self.w
        Hq, Hkv, hd = c.Hq, c.Hkv, c.hd

        def snap(name, t):
            if trace is not None:
                trace[name] = t.clone()

        def done(name):
            if mark is not None:
                mark(name)

        B.biv_embed_rmsnorm(w["embed"], win.tokens, w["l0.attn_norm"], self.x, self.h, c.eps)
        done("embed_rmsnorm")
        snap("x_in", self.x)
        for l in range(c.layers):
            snap(f"l{l}.h_attn", self.h)
            # QKV projection; its epilogue rotates q and k and writes k and v
            # straight into the cache rows of the window (the unrotated
            # projection is stored only when tracing)
            B.biv_gemm_qkv_rope(self.h, w[f"l{l}.wqkv_rope"], self.q, self.kc[l], self.vc[l], win.row_slot,
                                win.row_pos, c.rope_theta, K=self.rpg,
                                qkv_out=self.qkv if trace is not None else None)
            done(f"l{l}.qkv_rope")
            snap(f"l{l}.qkv", self.qkv)
            snap(f"l{l}.q", self.q)
            if trace is not None:
                trace[f"l{l}.kc"], trace[f"l{l}.vc"] = self.kc[l].clone(), self.vc[l].clone()
            B.biv_decode_attn_fixedsplit(self.q, self.kc[l], self.vc[l], win.row_slot, win.row_pos, self.o,
                                         self.rpg, self.workspace)
            done(f"l{l}.attention")
            snap(f"l{l}.o", self.o)
            B.biv_gemm_nosplitk(self.o.view(self.W, Hq * hd), w[f"l{l}.wo"], self.proj)
            done(f"l{l}.wo")
            snap(f"l{l}.attn_proj", self.proj)
            B.biv_add_rmsnorm(self.x, self.proj, w[f"l{l}.ffn_norm"], self.x, self.h, c.eps)
            done(f"l{l}.add_rmsnorm1")
            snap(f"l{l}.x_mid", self.x)
            snap(f"l{l}.h_ffn", self.h)
            B.biv_gemm_swiglu(self.h, w[f"l{l}.wgu_packed"], self.act)
            done(f"l{l}.gate_up_swiglu")
            snap(f"l{l}.act", self.act)
            B.biv_gemm_nosplitk(self.act, w[f"l{l}.wdown"], self.proj)
            done(f"l{l}.down")
            snap(f"l{l}.down", self.proj)
            last = l + 1 == c.layers
            gain = w["final_norm"] if last else w[f"l{l + 1}.attn_norm"]
            B.biv_add_rmsnorm(self.x, self.proj, gain, self.x, self.hidden if last else self.h, c.eps)
            done(f"l{l}.add_rmsnorm2")
            snap(f"l{l}.x_out", self.x)
        snap("hidden", self.hidden)

    def lm_head(self, win: Window) -> None:
        """fp32 logits (unfused), or logits (if kept) and the selected tokens."""
        if self.fused_select:
            B.biv_lm_head_gumbel(self.hidden, self.w["lm_head"], win.row_req, win.row_pos, self.seed,
                                 self.cfg.temperature, self.target, self.select_ws, logits=self.logits)
        else:
            B.biv_gemm_nosplitk(self.hidden, self.w["lm_head"], self.logits)

    def select_and_accept(self, win: Window) -> None:
        if not self.fused_select:
            B.biv_gumbel_argmax(self.logits, win.row_req, win.row_pos, self.seed, self.cfg.temperature,
                                self.target)
        N = self.accept_len.shape[0]
        B.biv_verify_accept(self.target, win.draft, win.p0, N, self.rpg, self.accept_len, self.new_len)

    def lm_head_accept(self, win: Window) -> None:
        """Tokens, accept lengths and new lengths from the final hidden rows."""
        if self.fused_select:
            # LM head with the selection in its epilogue, then winners + accept in one kernel
            B.biv_lm_head_gumbel_accept(self.hidden, self.w["lm_head"], win.row_req, win.row_pos, self.seed,
                                        self.cfg.temperature, self.target, win.draft, win.p0,
                                        self.accept_len.shape[0], self.rpg, self.accept_len, self.new_len,
                                        self.select_ws, logits=self.logits)
        else:
            self.lm_head(win)
            self.select_and_accept(win)

    def step(self, win: Window, mark=None) -> None:
        self.forward(win, mark=mark)
        self.lm_head_accept(win)
        if mark is not None:
            mark("lm_head_select_accept")

    def prefill(self, win: Window) -> None:
        """Deterministic prefill ([DVR] para 3: the verifier's fixed-shape
        forward also produces the first token and the initial KV): the prompt
        is one window of one request, rows at positions 0..P-1, so every row's
        K/V lands in the cache and row P-1 selects the first new token
        (``target[P-1]``).  No accept step: there are no drafts."""
        self.forward(win)
        self.lm_head(win)
        if not self.fused_select:
            B.biv_gumbel_argmax(self.logits, win.row_req, win.row_pos, self.seed, self.cfg.temperature,
                                self.target)

    # -------------------------------------------------------- CUDA graphs
    def capture(self, win: Window, segments: bool = False):
        """Capture the step on ``win``'s (static) buffers.

        With ``segments`` the step is captured as two graphs -- the layers,
        then the LM head with selection and accept -- so the LM-head launch
        can be timed with events between replays.
        """
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step(win)            # warm-up outside capture (sets kernel attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        parts = [(self.forward, (win,)), (self.lm_head_accept, (win,))]
        if not segments:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(win)
            return g
        graphs = []
        for fn, args in parts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(*args)
            graphs.append(g)
        return graphs


def prefill_window(prompt, slot: int, req_id: int, device="cuda") -> Window:
    """The window of a prefill: one request, one row per prompt token at
    positions 0..P-1 of cache slot ``slot``."""
    prompt = torch.as_tensor(prompt, dtype=torch.int32)
    P = prompt.numel()
    win = make_window(1, P, prompt, torch.zeros(1, dtype=torch.int32), torch.tensor([req_id], dtype=torch.int32),
                      torch.zeros(P, dtype=torch.int32), device=device)
    win.row_slot.fill_(slot)
    return win


class PackedWindow:
    """A window whose six inputs are views of one device buffer, fed from one
    pinned host buffer: [tokens W | row_slot W | row_req W | row_pos W |
    draft W | p0 N] (int32), so one host-to-device copy moves a step's inputs."""

    def __init__(self, N: int, K: int, device="cuda"):
        W = N * K
        self.host = torch.empty(5 * W + N, dtype=torch.int32).pin_memory()
        self.dev = torch.empty(5 * W + N, dtype=torch.int32, device=device)
        v = [self.dev[i * W:(i + 1) * W] for i in range(5)]
        self.win = Window(tokens=v[0], row_slot=v[1], row_req=v[2], row_pos=v[3], draft=v[4], p0=self.dev[5 * W:])

    def set(self, win: Window) -> None:
        """Host copy of ``win``'s inputs (the next step's window)."""
        parts = [win.tokens, win.row_slot, win.row_req, win.row_pos, win.draft, win.p0]
        self.host.copy_(torch.cat([t.cpu() for t in parts]))


def capture_e2e(ver: DecoderVerifier, pw: PackedWindow, host_results: torch.Tensor):
    """One CUDA graph of a whole end-to-end step: the inputs' host-to-device
    copy (pinned), the verify step, the results' device-to-host copy (pinned
    ``host_results``, int32 [2N + W]).  Replay it, then synchronise."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pw.dev.copy_(pw.host, non_blocking=True)
        ver.step(pw.win)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pw.dev.copy_(pw.host, non_blocking=True)
        ver.step(pw.win)
        host_results.copy_(ver.results, non_blocking=True)
    return g


def make_window(N: int, K: int, tokens, p0, req_ids, draft, device="cuda") -> Window:
    """Build a request-major window (row r*K + j in slot r at position p0[r] + j)."""
    dev = torch.device(device)
    p0 = torch.as_tensor(p0, dtype=torch.int32)
    req_ids = torch.as_tensor(req_ids, dtype=torch.int32)
    r = torch.arange(N, dtype=torch.int32).repeat_interleave(K)
    j = torch.arange(K, dtype=torch.int32).repeat(N)
    i32 = lambda t: torch.as_tensor(t, dtype=torch.int32).to(dev).contiguous()
    return Window(tokens=i32(tokens), row_slot=i32(r), row_req=i32(req_ids[r.long()]),
                  row_pos=i32(p0[r.long()] + j), draft=i32(draft), p0=i32(p0))
