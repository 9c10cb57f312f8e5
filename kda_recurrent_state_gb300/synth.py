"""Seeded synthetic inputs shaped like the KDA workloads.

This module only draws random numbers (torch generators, fixed seeds).  It
holds none of the attention arithmetic, so both the CUDA path and the fp64
oracle can take their inputs from it: the same tensors (bytes) feed both.

Distributions (per tensor, i.i.d. unless stated):
  q, k      ~ N(0, 1), then L2-normalised over the key dimension for every
              (token, head); the caller owns this normalisation, the
              operator does not normalise.
  v         ~ N(0, 1)
  beta      = sigmoid(N(0, 1))                           (fp32)
  log_alpha = -Uniform(0.001, 0.1) per key channel     (fp32, "config" gates;
              head_gates draws one per (token, head) the same way)
              -Uniform(1e-5, 1e-3)                       ("slow" gates: the
              initial state and the chunk carry stay visible for thousands
              of tokens, so they are actually tested)
              -Uniform(0.15, 0.2)                        ("steep": a chunk's
              decay close to what the fp16 operand path factors)
              "mixed": key channels 0..63 fast, -Uniform(1, 10) (they forget
              within a few tokens; channels 0..3 exactly -30), channels
              64..127 slow as above: the per-channel forgetting the method
              exists for, beyond any per-chunk factoring of the decay
  state     ~ N(0, 0.02)                                (fp32)
"""
from __future__ import annotations

import math

import torch

SEED_BASE = 0x4B4441  # "KDA"


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _gates(shape, g, device, gate: str) -> torch.Tensor:
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    if gate == "mixed":  # per key channel (the last dimension)
        c = torch.arange(shape[-1], device=device)
        fast, slow = -(1.0 + 9.0 * u), -(1e-5 + (1e-3 - 1e-5) * u)
        la = torch.where(c < shape[-1] // 2, fast, slow)
        return torch.where(c < 4, torch.full_like(la, -30.0), la)
    lo, hi = {"config": (0.001, 0.1), "slow": (1e-5, 1e-3), "steep": (0.15, 0.2)}[gate]
    return -(lo + (hi - lo) * u)


def head_gates(lead: tuple, H: int, *, seed: int, device="cpu", gate: str = "config") -> torch.Tensor:
    """One log-decay per (token, head), ``lead + (H,)`` fp32, from the same distribution as the
    per-channel gates (the scalar gate of Gated DeltaNet)."""
    return _gates((*lead, H), _gen(device, seed), device, gate)


def token_tensors(lead: tuple, H: int, dk: int, dv: int, g, device, in_dtype, gate: str):
    """q, k, v, log_alpha, beta for token-major layouts ``lead + (H, d)``."""
    q = _unit_rows(torch.randn(*lead, H, dk, generator=g, device=device, dtype=torch.float32)).to(in_dtype)
    k = _unit_rows(torch.randn(*lead, H, dk, generator=g, device=device, dtype=torch.float32)).to(in_dtype)
    v = torch.randn(*lead, H, dv, generator=g, device=device, dtype=torch.float32).to(in_dtype)
    beta = torch.sigmoid(torch.randn(*lead, H, generator=g, device=device, dtype=torch.float32))
    la = _gates((*lead, H, dk), g, device, gate)
    return q, k, v, la, beta


def prefill_inputs(B: int, T: int, H: int, dk: int = 128, dv: int = 128, *, seed: int, device="cpu",
                   in_dtype=torch.bfloat16, init: str = "zero", gate: str = "config") -> dict:
    """Batched prefill: q,k,v [B,T,H,d]; log_alpha [B,T,H,dk]; beta [B,T,H]; init_state [B,H,dk,dv] or None."""
    g = _gen(device, seed)
    q, k, v, la, beta = token_tensors((B, T), H, dk, dv, g, device, in_dtype, gate)
    S0 = None
    if init == "normal":
        S0 = 0.02 * torch.randn(B, H, dk, dv, generator=g, device=device, dtype=torch.float32)
    return dict(q=q, k=k, v=v, log_alpha=la, beta=beta, init_state=S0)


def varlen_lengths(N: int, lo: int, hi: int, seed: int) -> list:
    """N sequence lengths drawn log-uniform in [lo, hi] (host RNG, seeded)."""
    g = _gen("cpu", seed)
    u = torch.rand(N, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + (math.log(hi) - math.log(lo)) * float(x)))) for x in u]


def varlen_inputs(lengths: list, H: int, dk: int = 128, dv: int = 128, *, seed: int, device="cpu",
                  in_dtype=torch.bfloat16, resume_every: int = 2, gate: str = "config") -> dict:
    """Packed sequences: q,k,v [Ttot,H,d]; cu_seqlens int64 [N+1]; init_states [N,H,dk,dv]
    (sequences 0, resume_every, 2*resume_every, ... resume from N(0,0.02); the rest start at zero)."""
    g = _gen(device, seed)
    N = len(lengths)
    Ttot = int(sum(lengths))
    q, k, v, la, beta = token_tensors((Ttot,), H, dk, dv, g, device, in_dtype, gate)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    S0 = torch.zeros(N, H, dk, dv, device=device, dtype=torch.float32)
    for s in range(0, N, max(1, resume_every)):
        S0[s] = 0.02 * torch.randn(H, dk, dv, generator=g, device=device, dtype=torch.float32)
    return dict(q=q, k=k, v=v, log_alpha=la, beta=beta, init_states=S0,
                cu_seqlens=torch.tensor(cu, dtype=torch.int64, device=device))


def decode_inputs(Bs: int, H: int, dk: int = 128, dv: int = 128, *, seed: int, steps: int, device="cpu",
                  in_dtype=torch.bfloat16, gate: str = "config") -> dict:
    """Decode: resident state [Bs,H,dk,dv] ~ N(0,0.02) and ``steps`` fresh token sets
    q,k,v [steps,Bs,H,d]; log_alpha [steps,Bs,H,dk]; beta [steps,Bs,H]."""
    g = _gen(device, seed)
    state = 0.02 * torch.randn(Bs, H, dk, dv, generator=g, device=device, dtype=torch.float32)
    q, k, v, la, beta = token_tensors((steps, Bs), H, dk, dv, g, device, in_dtype, gate)
    return dict(state=state, q=q, k=k, v=v, log_alpha=la, beta=beta)
