"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

# bf16 kernel outputs vs the fp64 oracle: |err| <= 2e-2 * max(1, |ref|).
BF16_RTOL = 2e-2


def assert_close(got, ref, tol=BF16_RTOL, what=""):
    g = got.detach().float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    bound = tol * np.maximum(1.0, np.abs(r))
    err = np.abs(g - r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} elements out of tolerance; worst at {i}: "
                             f"got {g[i]!r} ref {r[i]!r}")
    return float((err / np.maximum(1.0, np.abs(r))).max()) if err.size else 0.0


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw bit pattern of a tensor (bitwise comparison, NaN-safe)."""
    t = t.detach().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.shape == b.shape and bool(torch.equal(bits(a), bits(b)))


def dev(t, device="cuda"):
    return t.to(device).contiguous()


# --------------------------------------------------- end-to-end tolerance
# The GPU composition and the oracle's (nearest-bf16 storage) both store
# bf16 at the same points but round slightly different values there (fp32
# accumulation on the GPU, fp64 in the oracle), so a correct GPU differs from
# the oracle by at most one bf16 ulp per stored element and the difference
# propagates to the logits.  The oracle composition that rounds every stored
# element in a random direction (one ulp off at about half of all elements
# of every storage point) bounds that drift; the tolerance is twice the
# largest drift of three such compositions, row by row.
E2E_SEEDS = (1, 2, 3)


def e2e_logit_envelope(orc, tokens, row_slot, row_pos, seeds=E2E_SEEDS):
    """(oracle logits with nearest-bf16 storage, per-row logit tolerance)."""
    outs = [orc.forward(tokens, row_slot, row_pos, storage="bf16_random", rng=np.random.default_rng(s))["logits"]
            for s in seeds]
    # last, so that the oracle's cache rows end with the nearest-bf16 values
    ref = orc.forward(tokens, row_slot, row_pos, storage="bf16")["logits"]
    env = np.max([np.abs(o - ref).max(axis=1) for o in outs], axis=0)
    return ref, 2.0 * env


def check_end_to_end(gpu_logits, gpu_tokens, ref_logits, tol_rows, row_req, row_pos, seed, T, what=""):
    """Logits within the per-row envelope; every token that differs from the
    oracle's selection on the oracle's logits sits on a row whose oracle key
    gap (the oracle's token's key minus the GPU token's key, both under the
    oracle's logits) is bridged by the two logits' drift -- at most
    invT (|dx_a| + |dx_b|) <= 2 invT tol_row, plus fp32 key rounding.
    Returns the number of rows whose tokens agree."""
    import oracle
    g = np.asarray(gpu_logits, np.float64)
    drift = np.abs(g - ref_logits)
    row_drift = drift.max(axis=1)
    bad = np.nonzero(row_drift > tol_rows)[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows drift past the envelope; worst row {bad[0]}: "
                           f"{row_drift[bad[0]]:.4g} > {tol_rows[bad[0]]:.4g}")
    rq, rp = np.asarray(row_req), np.asarray(row_pos)
    otg = oracle.gumbel_argmax(ref_logits.astype(np.float32), rq, rp, seed, T)
    tgt = np.asarray(gpu_tokens)
    diff = np.nonzero(otg != tgt)[0]
    if diff.size:
        invT = 1.0 if T == 0 else float(np.float32(1.0) / np.float32(T))
        keys = oracle.gumbel_keys(ref_logits[diff].astype(np.float32), rq[diff], rp[diff], seed, T)
        for i, r in enumerate(diff):
            a, b = int(tgt[r]), int(otg[r])
            gap = float(keys[i, b]) - float(keys[i, a])
            slack = 4.0 * float(np.spacing(np.float32(max(abs(keys[i, a]), abs(keys[i, b])))))
            bridged = invT * (drift[r, a] + drift[r, b]) + slack
            assert 0.0 <= gap <= bridged, f"{what}: row {r} token {a} vs oracle {b}: gap {gap:.4g} > {bridged:.4g}"
            assert gap <= 2.0 * invT * tol_rows[r] + slack
    return int(tgt.size - diff.size)
