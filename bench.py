"""Benchmark: verified tokens/s of the batch-invariant verify step.

Workload: the random-init 2-layer decoder verifier (d=1024, 8 query / 2 KV
heads of 128, SwiGLU 2816, vocab 32000, bf16 weights ~N(0, 0.02)), one
window of N=8 requests x K=8 tokens (W = 64 rows), per-request contexts
~U[128, 2048], fixed KV split 256, drafts with a 30% random-token error
rate, Gumbel selection at T=0.7.  One step = the whole hot path: embed,
2 x (RMSNorm, QKV GEMM, RoPE, KV overwrite, fixed-split attention, Wo GEMM,
residual, RMSNorm, gate/up GEMM, SwiGLU, down GEMM, residual), RMSNorm,
LM-head GEMM (fp32 logits), Gumbel-max selection, coupled accept.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): the path shards by request, so each rank runs its own
replica window (weak scaling, no collective on the data path); value is the
rows of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the plain C++ reference) on the same
workload, one window row per step, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified tok/s at W=N·K, batch-invariant; % of bf16 tensor-core / HBM roofline"
UNIT = "verified tok/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--gemm-sweep", action="store_true",
                   help="instead of the step bench: no-split-K GEMM vs cuBLAS on the Llama-3-8B shapes")
    p.add_argument("--kernel-sweep", action="store_true",
                   help="instead of the step bench: HBM GB/s of RMSNorm, attention and Gumbel-max at full sizes")
    p.add_argument("--c4-steps", action="store_true",
                   help="instead of the step bench: verified tok/s of whole verify steps on the Llama-3-8B-shaped "
                        "layer + LM head at the verifier sweep's windows (N x K = 8x4, 32x8, 64x16)")
    p.add_argument("--profile-case", choices=["attn16", "select1024"],
                   help="run one small case twice, for a profiler capture: attention on 16 requests x 16 rows "
                        "(C4 recipe) or selection on 1024 rows (C5 recipe, T = 0.7 then T = 0)")
    return p.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def workload_config(cfg):
    return {"workload": "2-layer decoder verifier d1024 8q/2kv hd128 ffn2816 vocab32000 (random init)",
            "N": cfg.N, "K": cfg.K, "W": cfg.W, "layers": cfg.layers, "d": cfg.d, "vocab": cfg.vocab,
            "ctx": f"U[{cfg.ctx_lo},{cfg.ctx_hi}]", "kv_split": cfg.kv_split, "temperature": cfg.temperature,
            "draft_error_rate": cfg.draft_err, "l2": "flushed between timed steps (256 MiB write, outside the step events)"}


# ------------------------------------------------------------------ setup
def build_problem(cfg, device, rank=0):
    """The rank's own window: requests rank*N .. rank*N + N - 1 of the job,
    with their own contexts, caches and drafts (weak scaling)."""
    from invariant_verify_gb300 import replicas, synth
    from invariant_verify_gb300.verifier import DecoderVerifier, make_window
    w = synth.decoder_weights(cfg)
    ctx = synth.context_lengths(cfg, cfg.N, seed=cfg.seed + 100 + rank)
    max_len = int(ctx.max()) + 64
    caches = synth.kv_cache(cfg.N, cfg.Hkv, max_len, cfg.hd, ctx, seed=cfg.seed + 200 + rank,
                            layers=cfg.layers)
    ver = DecoderVerifier(cfg, w, caches, cfg.N, max_len, cfg.W, cfg.K, device=device, fused_select=True,
                          keep_logits=False)
    g = synth.generator(cfg.seed + 300 + rank)
    N, K = cfg.N, cfg.K
    last = torch.randint(0, cfg.vocab, (N,), generator=g, dtype=torch.int64).to(torch.int32)
    mask, ids = synth.draft_errors((N, K), cfg.draft_err, cfg.vocab, seed=cfg.seed + 400 + rank)
    req = replicas.request_ids(replicas.rank_requests(N, rank))
    # A drafter that is right 70% of the time: fix d_1..d_K one position at a
    # time from the verifier's own selections (d_j feeds row j).
    drafts = torch.zeros(N, K, dtype=torch.int32)
    for j in range(K):
        tokens = torch.cat([last[:, None], drafts[:, :-1]], dim=1)
        win = make_window(N, K, tokens.reshape(-1), ctx, req, drafts.reshape(-1), device=device)
        ver.step(win)
        tgt = ver.target.view(N, K)[:, j].cpu()
        drafts[:, j] = torch.where(mask[:, j], ids[:, j], tgt)
    tokens = torch.cat([last[:, None], drafts[:, :-1]], dim=1)
    win = make_window(N, K, tokens.reshape(-1), ctx, req, drafts.reshape(-1), device=device)
    return ver, win, w, caches, max_len, ctx


def clock_sampler_start(path):
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"],
                             stdout=f, stderr=subprocess.DEVNULL)
        return p, f
    except Exception:
        return None, None


def clock_sampler_stop(p, f, path, gpu_index):
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except Exception:
        p.kill()
    f.close()
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != gpu_index:
            continue
        try:
            sm.append(float(parts[1]))
            mx = float(parts[2])
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def lm_head_traffic():
    """Per-launch DRAM bytes of the fused LM-head/selection kernel from the
    committed ncu summary, or None when the kernel source changed since that
    capture."""
    path = os.path.join(ROOT, "profiles", "lmhead_select_fused_decoder2.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    return float(m.group(1)) if kernel_source_sha256().startswith(h.group(1)) else None


def kernel_source_sha256():
    """Hash of the sources the fused LM-head/selection kernel is built from."""
    csrc = os.path.join(ROOT, "invariant_verify_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("biv_gemm.cu", "biv_gumbel.cuh", "biv_common.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


def marked_graphs(ver, win, n):
    """``n`` graphs of the whole step, each with its own pair of timing events
    recorded as graph nodes immediately before and after the LM-head launch;
    None where this PyTorch cannot record events inside a graph."""
    try:
        pool = []
        for _ in range(n):
            ea = torch.cuda.Event(enable_timing=True, external=True)
            eb = torch.cuda.Event(enable_timing=True, external=True)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                ver.forward(win)
                ea.record()
                ver.lm_head_accept(win)
                eb.record()
            pool.append((g, ea, eb))
        g, ea, eb = pool[0]
        g.replay()
        eb.synchronize()
        ea.elapsed_time(eb)
        return pool
    except (TypeError, RuntimeError) as exc:
        print(f"bench: no event nodes in graphs ({exc}); timing the LM head between graph segments",
              file=sys.stderr)
        torch.cuda.synchronize()
        return None


# --------------------------------------------------------------- our arm
def run_ours(args):
    import torch.distributed as dist
    from invariant_verify_gb300 import replicas, synth
    import __graft_entry__
    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    cfg = synth.DECODER2
    ver, win, w_cpu, caches_cpu, max_len, ctx = build_problem(cfg, device, rank=rank)
    full_graph = ver.capture(win, segments=False)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    K = args.steps
    # Each timed step replays one graph of the whole step.  The LM-head launch
    # is bracketed by event-record nodes inside that graph (a pool of graphs,
    # each with its own event pair, read back once its replay has finished);
    # where event nodes are unavailable the step is replayed as two graphs
    # with events between them.
    pool = marked_graphs(ver, win, min(K, 16))
    lm_timing = "event-record nodes around the LM-head launch inside the step graph"
    if pool is None:
        segs = ver.capture(win, segments=True)
        lm_timing = "events between graph segments (layers | LM head + selection + accept)"

    def one_step(i):
        if pool is None:
            segs[0].replay()
            seg_ev[i][0].record(stream)
            segs[1].replay()
            seg_ev[i][1].record(stream)
        else:
            pool[i % len(pool)][0].replay()

    seg_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)] if pool is None else None
    for i in range(max(3, args.warmup)):
        flush.zero_()
        one_step(i % K)
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    lm_ms = []
    out_dir = os.environ.get("BIV_BENCH_OUT_DIR", "/tmp")      # where the raw clock samples go
    clk_path = os.path.join(out_dir if os.path.isdir(out_dir) else "/tmp", f"bench_clocks_rank{rank}.csv")
    sampler, sf = clock_sampler_start(clk_path) if local == 0 else (None, None)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        if pool is not None and i >= len(pool):
            _, ea, eb = pool[i % len(pool)]
            eb.synchronize()                 # that graph's previous replay is done
            lm_ms.append(ea.elapsed_time(eb))
        flush.zero_()
        e = ev[i]
        e[0].record(stream)
        one_step(i)
        e[1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    clocks = clock_sampler_stop(sampler, sf, clk_path, local)
    if pool is not None:
        for i in range(max(0, K - len(pool)), K):
            _, ea, eb = pool[i % len(pool)]
            lm_ms.append(ea.elapsed_time(eb))
    else:
        lm_ms = [a.elapsed_time(b) for a, b in seg_ev]
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    tot_ms = replicas.slowest(float(sum(step_ms)), device=device)
    ms_per_step = tot_ms / K
    value = cfg.W * world * K / (tot_ms / 1e3)
    committed = int(ver.accept_len.sum().item())

    # roofline of the dominant kernel (LM-head GEMM, HBM-bound at W=64)
    hbm, bf16, src = peaks()
    M, N, Kd = cfg.W, cfg.vocab, cfg.d
    # weights + activations in, request ids / positions in, tokens out (the
    # logits stay in TMEM; the per-tile winners and the accept's few bytes
    # per request are not counted)
    lm_bytes = 2 * N * Kd + 2 * M * Kd + 12 * M
    lm_avg_s = statistics.mean(lm_ms) / 1e3
    achieved = lm_bytes / lm_avg_s / 1e9
    roofline = {"kernel": "gemm_nosplitk_kernel<3> + winners_accept_kernel (LM head M=64 N=32000 K=1024 with "
                          "the Gumbel-max selection in its epilogue, then the per-row winners and the accept)",
                "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                "traffic": lm_head_traffic(), "algorithmic_bytes": lm_bytes,
                "avg_launch_us": round(lm_avg_s * 1e6, 2), "launch_timing": lm_timing}
    step_bytes, step_flops = step_work(cfg, ctx)
    step_roof_us = max(step_bytes / (hbm * 1e9), step_flops / (bf16 * 1e12)) * 1e6

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(ver, win, full_graph, flush, cfg, max(50, min(K, 2000)), world, device)

    out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
           "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": workload_config(cfg) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
           "roofline": roofline,
           "step_roofline": {"bytes": step_bytes, "flops": step_flops, "lower_bound_us": round(step_roof_us, 2),
                             "frac": round(step_roof_us / (ms_per_step * 1e3), 4)},
           "committed_tok_per_s": round(committed * world * K / (tot_ms / 1e3), 1),
           "gpu_launches": ver.launches_per_step * K,
           "timed_region_wall_s": round(wall, 3),
           "clocks": clocks, "e2e": e2e}
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(cfg, w_cpu, caches_cpu, max_len, win, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def step_work(cfg, ctx):
    """Algorithmic bytes and flops of one step (weights once, KV read,
    activations ignored; the logits never reach HBM)."""
    W, d, F, V, hd = cfg.W, cfg.d, cfg.ffn, cfg.vocab, cfg.hd
    per_layer_w = (cfg.qkv_n * d + d * cfg.Hq * hd + 2 * F * d + d * F) * 2
    weights = cfg.layers * per_layer_w + V * d * 2
    kv = sum(2 * 2 * cfg.Hkv * (int(c) + cfg.K) * hd for c in ctx) * cfg.layers
    logits = 0
    flops = 2 * W * (cfg.layers * per_layer_w // 2 + V * d)
    flops += cfg.layers * sum(4 * cfg.Hq * cfg.K * (int(c) + cfg.K) * hd for c in ctx)
    return weights + kv + logits, flops


def run_e2e(ver, win, graph, flush, cfg, K, world, device):
    """Same metric through the public API with host buffers: each step copies
    the window's inputs from pinned host memory (one copy of the packed
    inputs), runs the step, and reads the accept lengths, rollback points and
    selected tokens back (one copy of the packed results) -- the three as
    nodes of one CUDA graph, replayed and synchronised per step."""
    from invariant_verify_gb300.verifier import PackedWindow, capture_e2e
    pw = PackedWindow(cfg.N, cfg.K, device=device)
    pw.set(win)
    host_out = torch.empty_like(ver.results, device="cpu").pin_memory()
    g = capture_e2e(ver, pw, host_out)
    h2d = pw.host.numel() * pw.host.element_size()
    d2h = host_out.numel() * host_out.element_size()
    stream = torch.cuda.current_stream()
    total = 0.0
    for i in range(K + 5):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        stream.synchronize()
        if i >= 5:
            total += time.perf_counter() - t0
    value = cfg.W * world * K / total
    return {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": K, "ms_per_step": round(total / K * 1e3, 5),
            "how": "one CUDA graph per step: pinned H2D of the packed window inputs, the step, D2H of the packed "
                   "accept_len/new_len/tokens; host wall time per step including the synchronisation"}


# ---------------------------------------------------------- kernel sweep
def _time_us(fn, reps=20, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
    for i in range(reps):
        ev[2 * i].record()
        fn()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    return statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps)) * 1e3


def run_kernel_sweep(args):
    """Achieved HBM bandwidth of the bandwidth-bound kernels at sizes far above
    L2 (inputs > 129 MB, so no flush is needed between launches): RMSNorm over
    [32768, 4096] bf16, the selection workload (fp32 [4096, 152064], T = 0.7),
    and the fixed-split attention of the verifier sweep's largest window
    (64 requests x 16 rows, Llama-3-8B heads, lognormal contexts)."""
    from invariant_verify_gb300 import abi as B
    from invariant_verify_gb300 import synth
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    hbm, _, src = peaks()
    out = []

    def line(kernel, workload, nbytes, us):
        gbs = nbytes / us / 1e3
        out.append({"kernel": kernel, "workload": workload, "algorithmic_bytes": int(nbytes), "us": round(us, 2),
                    "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4), "peak_source": src})
        print(json.dumps(out[-1]), flush=True)

    rows, d = 32768, 4096
    x = synth.bf16_normal_device((rows, d), 1.0, 7)
    w = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    line("rmsnorm_kernel", "rmsnorm bf16 [32768, 4096]", 4 * rows * d + 2 * d,
         _time_us(lambda: B.biv_rmsnorm(x, w, y, 1e-6)))
    del x, y

    cfg = synth.SELECT
    logits = synth.select_logits_device(cfg)
    R = cfg.R
    req = (torch.arange(R, dtype=torch.int32, device="cuda") // cfg.K) * 7 + 3
    pos = (torch.arange(R, dtype=torch.int32, device="cuda") % cfg.K) + 1000
    tok = torch.empty(R, dtype=torch.int32, device="cuda")
    line("gumbel_stream_kernel", "select fp32 [4096, 152064], T=0.7, 90% peaked rows",
         4 * R * cfg.vocab + 12 * R, _time_us(lambda: B.biv_gumbel_argmax(logits, req, pos, synth.PHILOX_SEED, 0.7, tok)))
    line("gumbel_stream_kernel", "select fp32 [4096, 152064], T=0 (greedy)",
         4 * R * cfg.vocab + 12 * R, _time_us(lambda: B.biv_gumbel_argmax(logits, req, pos, synth.PHILOX_SEED, 0.0, tok)))
    del logits

    sw = synth.SWEEP
    N, K = 64, 16
    W = N * K
    ctx = synth.context_lengths(sw, N, seed=123)
    max_len = int(ctx.max()) + K + 8
    kc, vc = synth.kv_cache_device(N, sw.Hkv, max_len, sw.hd, ctx, seed=124, layers=1)[0]
    q = synth.bf16_normal_device((W, sw.Hq, sw.hd), 1.0, 125)
    o = torch.empty_like(q)
    slot = torch.arange(N, dtype=torch.int32, device="cuda").repeat_interleave(K)
    rpos = (ctx.cuda().repeat_interleave(K) + torch.arange(K, device="cuda").repeat(N)).to(torch.int32)
    ws = torch.empty(B.biv_decode_attn_workspace_size(W, sw.Hq, max_len), dtype=torch.uint8, device="cuda")
    kv_bytes = sum(2 * 2 * sw.Hkv * (int(c) + K) * sw.hd for c in ctx)
    line("attn_tc_kernel + attn_combine_kernel",
         f"attention W={W} (64 x 16), Hq 32 / Hkv 8, lognormal ctx mean {float(ctx.float().mean()):.0f}",
         kv_bytes + 2 * 2 * W * sw.Hq * sw.hd,
         _time_us(lambda: B.biv_decode_attn_fixedsplit(q, kc, vc, slot, rpos, o, K, ws)))
    return out


# ------------------------------------------------------------ GEMM sweep
def run_gemm_sweep(args):
    """TFLOP/s and HBM GB/s of the no-split-K GEMM against cuBLAS's default
    (torch.matmul, free to split K) on the Llama-3-8B-shaped weights, and how
    many output rows cuBLAS changes bitwise when the same rows are computed
    at another M (the cost and the need for invariance)."""
    from invariant_verify_gb300 import abi as B
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    hbm, bf16, _ = peaks()
    shapes = {"qkv": (6144, 4096), "wo": (4096, 4096), "gate_up": (28672, 4096), "down": (4096, 14336),
              "lm_head": (128256, 4096)}
    Ms = [1, 8, 32, 64, 128, 256, 512, 1024]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    rows = []
    for name, (N, K) in shapes.items():
        g = torch.Generator(device="cuda").manual_seed(N + K)
        Bw = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        A = torch.randn(max(Ms), K, device="cuda", generator=g).to(torch.bfloat16)
        ref_ours = torch.empty(max(Ms), N, device="cuda", dtype=torch.bfloat16)
        B.biv_gemm_nosplitk(A, Bw, ref_ours)
        ref_cublas = A @ Bw.t()
        for M in Ms:
            a = A[:M].contiguous()
            c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
            times = {}
            for impl in ("ours", "cublas"):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * 20)]
                for i in range(23):
                    flush.zero_()
                    if i >= 3:
                        ev[2 * (i - 3)].record()
                    if impl == "ours":
                        B.biv_gemm_nosplitk(a, Bw, c)
                    else:
                        torch.matmul(a, Bw.t(), out=c)
                    if i >= 3:
                        ev[2 * (i - 3) + 1].record()
                torch.cuda.synchronize()
                times[impl] = statistics.median(ev[2 * j].elapsed_time(ev[2 * j + 1]) for j in range(20)) / 1e3
            ours_rows = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
            B.biv_gemm_nosplitk(a, Bw, ours_rows)
            diff_ours = int((ours_rows.view(torch.int16) != ref_ours[:M].view(torch.int16)).any(dim=1).sum())
            diff_cublas = int((torch.matmul(a, Bw.t()).view(torch.int16) !=
                               ref_cublas[:M].view(torch.int16)).any(dim=1).sum())
            flops = 2.0 * M * N * K
            byts = 2.0 * N * K + 2.0 * M * K + 2.0 * M * N
            rows.append({"gemm": name, "M": M, "N": N, "K": K,
                         "ours_us": round(times["ours"] * 1e6, 2), "cublas_us": round(times["cublas"] * 1e6, 2),
                         "ours_tflops": round(flops / times["ours"] / 1e12, 1),
                         "cublas_tflops": round(flops / times["cublas"] / 1e12, 1),
                         "ours_gbs": round(byts / times["ours"] / 1e9, 1),
                         "ours_frac_hbm": round(byts / times["ours"] / 1e9 / hbm, 3),
                         "ours_frac_tensor": round(flops / times["ours"] / 1e12 / bf16, 3),
                         "rows_differing_vs_M1024": {"ours": diff_ours, "cublas": diff_cublas}})
            print(json.dumps(rows[-1]), flush=True)
    return rows


# ------------------------------------------------------- CPU oracle timing
def oracle_rows_per_second(cfg, w_cpu, caches_cpu, max_len, win, seconds, max_steps=None, warmup=0):
    import oracle
    from oracle.model import OracleDecoder
    orc = OracleDecoder(cfg, w_cpu, caches_cpu, cfg.N, max_len)
    tokens = win.tokens.cpu().numpy()
    slot = win.row_slot.cpu().numpy()
    req = win.row_req.cpu().numpy()
    pos = win.row_pos.cpu().numpy()
    # The window's own K/V rows must be in the cache before single rows are
    # verified: one full oracle forward writes them (not timed).
    orc.forward(tokens, slot, pos)
    W = tokens.size
    done, spent, i = 0, 0.0, 0
    while True:
        r = i % W
        t0 = time.perf_counter()
        out = orc.forward(tokens[r:r + 1], slot[r:r + 1], pos[r:r + 1])
        oracle.gumbel_argmax(out["logits"].astype(np.float32), req[r:r + 1], pos[r:r + 1], 0x1234_5678_9ABC_DEF0,
                             cfg.temperature)
        dt = time.perf_counter() - t0
        i += 1
        if i <= warmup:
            continue
        done += 1
        spent += dt
        if (max_steps is not None and done >= max_steps) or (max_steps is None and spent >= seconds):
            break
    import oracle as _o
    return done / spent, done, spent, _o.num_threads()


def cpu_baseline(cfg, w_cpu, caches_cpu, max_len, win, seconds):
    v, n, spent, cores = oracle_rows_per_second(cfg, w_cpu, caches_cpu, max_len, win, seconds)
    return {"value": round(v, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} window rows verified one at a time (all layers + LM head + selection, fp64) "
                      f"in {spent:.1f} s on {cores} host threads"}


# --------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    from invariant_verify_gb300 import replicas, synth
    from invariant_verify_gb300.verifier import make_window
    from oracle import build as ob
    ob.build()
    cfg = synth.DECODER2
    w = synth.decoder_weights(cfg)
    ctx = synth.context_lengths(cfg, cfg.N, seed=cfg.seed + 100)
    max_len = int(ctx.max()) + 64
    caches = synth.kv_cache(cfg.N, cfg.Hkv, max_len, cfg.hd, ctx, seed=cfg.seed + 200, layers=cfg.layers)
    g = synth.generator(cfg.seed + 300)
    toks = torch.randint(0, cfg.vocab, (cfg.W,), generator=g, dtype=torch.int64).to(torch.int32)
    win = make_window(cfg.N, cfg.K, toks, ctx, replicas.request_ids(range(cfg.N)), toks, device="cpu")
    steps = max(1, args.steps)
    v, n, spent, cores = oracle_rows_per_second(cfg, w, caches, max_len, win, 0.0, max_steps=steps,
                                                warmup=max(0, min(args.warmup, 3)))
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
           "steps": n, "warmup": args.warmup, "ms_per_step": round(spent / n * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(cfg) | {"parallelism": "host cores"},
           "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": "one window row per step (all layers + LM head + selection, fp64)"},
           "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_c4_steps(args):
    """Whole verify steps (embed + RMSNorm, one Llama-3-8B-shaped layer, LM
    head over 128256 tokens with the fused selection, winners + accept) at the
    verifier sweep's windows, lognormal contexts.  Each step is one CUDA graph
    replay; the weights (1.49 GB) and KV caches exceed L2, so no flush is
    needed.  Device-timed with events around each replay."""
    from invariant_verify_gb300 import synth
    from invariant_verify_gb300.verifier import DecoderVerifier, make_window
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    hbm, bf16, src = peaks()
    cfg = synth.SWEEP
    w = synth.decoder_weights_device(cfg)
    for N, K in ((8, 4), (32, 8), (64, 16)):
        W = N * K
        ctx = synth.context_lengths(cfg, N, seed=40 + N)
        max_len = int(ctx.max()) + K + 16
        caches = synth.kv_cache_device(N, cfg.Hkv, max_len, cfg.hd, ctx, seed=41 + N, layers=cfg.layers)
        ver = DecoderVerifier(cfg, w, caches, N, max_len, W, K, keep_logits=False)
        req = torch.arange(N, dtype=torch.int32) * 31 + 1
        toks = torch.randint(0, cfg.vocab, (W,), generator=synth.generator(43), dtype=torch.int64).to(torch.int32)
        win = make_window(N, K, toks, ctx, req, toks)
        g = ver.capture(win)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        n = 20
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
        kv = sum(2 * 2 * cfg.Hkv * (int(c) + K) * cfg.hd for c in ctx)
        wbytes = sum(t.numel() * t.element_size() for k, t in w.items() if k != "embed")
        flops = 2 * W * (wbytes // 2) + 4 * cfg.Hq * cfg.hd * sum(int(c) + K for c in ctx) * K
        lb = max((wbytes + kv) / (hbm * 1e9), flops / (bf16 * 1e12)) * 1e6
        print(json.dumps({"workload": f"C4 verify step N={N} K={K} W={W}, Llama-3-8B-shaped layer + LM head "
                                      f"(vocab {cfg.vocab}), lognormal ctx mean {float(ctx.float().mean()):.0f}",
                          "us_per_step": round(us, 1), "verified_tok_per_s": round(W / us * 1e6, 1),
                          "lower_bound_us": round(lb, 1), "frac_of_roofline": round(lb / us, 4),
                          "gpu_launches_per_step": ver.launches_per_step, "peak_source": src}), flush=True)
        del ver, caches, g
        torch.cuda.empty_cache()


def run_profile_case(args):
    """A small case of one kernel, launched twice (the second launch is the
    one to capture): inputs above L2 size, a few hundred MB on the device."""
    import dataclasses
    from invariant_verify_gb300 import abi as B
    from invariant_verify_gb300 import synth
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    if args.profile_case == "attn16":
        sw = synth.SWEEP
        N, K = 16, 16
        W = N * K
        ctx = synth.context_lengths(sw, N, seed=123)
        max_len = int(ctx.max()) + K + 8
        kc, vc = synth.kv_cache_device(N, sw.Hkv, max_len, sw.hd, ctx, seed=124, layers=1)[0]
        q = synth.bf16_normal_device((W, sw.Hq, sw.hd), 1.0, 125)
        o = torch.empty_like(q)
        slot = torch.arange(N, dtype=torch.int32, device="cuda").repeat_interleave(K)
        rpos = (ctx.cuda().repeat_interleave(K) + torch.arange(K, device="cuda").repeat(N)).to(torch.int32)
        ws = torch.empty(B.biv_decode_attn_workspace_size(W, sw.Hq, max_len), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            B.biv_decode_attn_fixedsplit(q, kc, vc, slot, rpos, o, K, ws)
        kv = sum(2 * 2 * sw.Hkv * (int(c) + K) * sw.hd for c in ctx)
        print(json.dumps({"case": "attn16", "kv_bytes": kv, "ctx_mean": float(ctx.float().mean())}))
    else:
        cfg = dataclasses.replace(synth.SELECT, requests=128)
        logits = synth.select_logits_device(cfg)
        R = cfg.R
        req = (torch.arange(R, dtype=torch.int32, device="cuda") // cfg.K) * 7 + 3
        pos = (torch.arange(R, dtype=torch.int32, device="cuda") % cfg.K) + 1000
        tok = torch.empty(R, dtype=torch.int32, device="cuda")
        for T in (0.7, 0.0):
            B.biv_gumbel_argmax(logits, req, pos, synth.PHILOX_SEED, T, tok)
        print(json.dumps({"case": "select1024", "rows": R, "vocab": cfg.vocab}))
    torch.cuda.synchronize()


if __name__ == "__main__":
    a = parse()
    if a.profile_case:
        run_profile_case(a)
    elif a.c4_steps:
        run_c4_steps(a)
    elif a.gemm_sweep:
        run_gemm_sweep(a)
    elif a.kernel_sweep:
        run_kernel_sweep(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
