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
