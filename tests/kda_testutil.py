"""Helpers shared by the GPU parity tests: layout conversion to the oracle's
head-major fp64 arrays and the error metrics.  No KDA arithmetic here."""
import numpy as np
import torch

# Tolerances for floating-point parity against the fp64 oracle (outputs and states).
REL_L2 = 2e-3
MAX_ABS = 1e-2


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def batch_heads(t: torch.Tensor, pairs):
    """[B,T,H,d] (or [B,T,H]) -> [n,T,d] (or [n,T]) for the listed (b,h) pairs."""
    return np.stack([np64(t[b, :, h]) for b, h in pairs])


def packed_heads(t: torch.Tensor, start: int, end: int, heads):
    """[Ttot,H,d] (or [Ttot,H]) -> [n,T,d] for tokens [start,end) and the listed heads."""
    return np.stack([np64(t[start:end, h]) for h in heads])


def errors(got, ref):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    mx = float(np.abs(g - r).max()) if g.size else 0.0
    return rel, mx


def assert_close(got, ref, what=""):
    rel, mx = errors(got, ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel-L2 {rel:.3e} (<= {REL_L2}), max-abs {mx:.3e} (<= {MAX_ABS})"
    return rel, mx
