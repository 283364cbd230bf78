"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module only draws random numbers and rounds them to bf16. It holds none of
the attention method's arithmetic (no mask, no softmax, no statistics).

Recipe (one ``torch.Generator`` seeded per workload, draws in this order):
  1. Q  = N(0, 1)  of shape [B, H, N, D]
  2. Z  = N(0, 1)  of shape [B, H, N, D]        (key noise)
  3. mu = s * N(0, 1) of shape [B, H, 1, D]     (per-head key mean offset)
  4. V  = N(0, 1)  of shape [B, H, N, D]
  5. for every outlier head h (ascending) and every batch b: one token index
     j ~ U{0..N-1}; that key row (Z + mu) is multiplied by 20
  K = Z + mu; Q, K, V are rounded to bf16 (round to nearest even).

Pre-attention chain inputs (``make_prologue_inputs``, one generator seeded
per call, draws in this order):
  1. x     = N(0, 1) of shape [B, N, C]          (hidden states)
  2. w     = N(0, 1) / sqrt(C) of shape [3HD, C] (q, k, v projection rows)
  3. gamma = 1 + 0.1 N(0, 1) of shape [C]        (RMSNorm gain, fp32)
     or, with ``exact_gain``, 2^e with e ~ U{-1, 0, 1}, so that w * gamma is
     exactly representable in bf16
  x and w are rounded to bf16.

The pages' production activations and weights are not available; these draws
stand in for them with the shapes and structure the workload presets name.
"""
from __future__ import annotations

import torch

from .configs import Workload

OUTLIER_FACTOR = 20.0


def make_qkv(w: Workload, seed: int | None = None, dtype=torch.bfloat16):
    """Return (q, k, v) bf16 CPU tensors of shape [B, H, N, D], contiguous."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.H, w.N, w.D)
    q = torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    mu = torch.randn((w.B, w.H, 1, w.D), generator=g, dtype=torch.float32) * w.key_offset_scale
    v = torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
    k += mu
    for h in sorted(w.outlier_heads):
        for b in range(w.B):
            j = int(torch.randint(0, w.N, (1,), generator=g).item())
            k[b, h, j, :] *= OUTLIER_FACTOR
    k = k.to(dtype)
    return q, k, v


def make_prologue_inputs(B: int, N: int, C: int, H: int, D: int, seed: int = 0,
                         exact_gain: bool = False):
    """Return (x bf16 [B, N, C], w bf16 [3HD, C], gamma fp32 [C]) CPU tensors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((B, N, C), generator=g, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((3 * H * D, C), generator=g, dtype=torch.float32) * C ** -0.5).to(torch.bfloat16)
    if exact_gain:
        gamma = torch.pow(2.0, torch.randint(-1, 2, (C,), generator=g).to(torch.float32))
    else:
        gamma = 1.0 + 0.1 * torch.randn((C,), generator=g, dtype=torch.float32)
    return x, w, gamma


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (for the C oracle)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def bf16_to_f64(t: torch.Tensor):
    """Exact float64 numpy copy of a bf16 tensor."""
    return t.to(torch.float64).numpy()
