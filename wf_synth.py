"""Seeded synthetic inputs for the wavefront round.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path's
tests and benchmark.  It holds random-number generation only: no step of
the method (no RoPE, no mask, no attention, no schedule) lives here.

Every tensor is keyed by the coordinates the pages use to name a piece of
work, so both sides can regenerate the same values independently:

* ``qkv_raw(seed, chunk, stage, layer, ...)``: the raw (pre-RoPE) Q/K/V that
  the QKV projection of task (chunk, stage) produces at one layer.  Stage S is
  the store pass.  Layout ``[tokens, 3, heads, head_dim]`` (token-major, the
  order a QKV projection writes).

The distributions follow the workloads the pages describe (Wan2.1-shaped
chunks of 3 latent frames; random-initialised weights): N(0, 1) scaled by a
caller-chosen factor (1/sqrt(head_dim) for the bf16 attention workload).
Values are rounded to the storage dtype *here*, so the oracle widens exactly
the numbers the GPU reads.
"""

from __future__ import annotations

import torch

__all__ = ["key_of", "qkv_raw", "normal"]


def key_of(seed: int, *coords: int) -> int:
    """Deterministic 63-bit key from a seed and integer coordinates.

    A plain polynomial mix (splitmix64 finaliser applied at each step); the
    only requirement is that distinct coordinate tuples give distinct
    generator seeds for the small ranges used here.
    """
    x = (seed & 0xFFFFFFFFFFFFFFFF) ^ 0x9E3779B97F4A7C15
    for c in coords:
        x = (x + (c & 0xFFFFFFFF) + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def normal(key: int, shape, scale: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """N(0, scale^2) samples on the CPU from a generator seeded with ``key``,
    rounded to ``dtype`` (returned in that dtype)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(key))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def qkv_raw(seed: int, chunk: int, stage: int, layer: int, n_tokens: int,
            heads: int, head_dim: int, scale: float = 1.0,
            dtype=torch.float32) -> torch.Tensor:
    """Raw Q/K/V of task (chunk, stage) at ``layer``: ``[n_tokens, 3, heads, head_dim]``."""
    return normal(key_of(seed, 1, chunk, stage, layer),
                  (n_tokens, 3, heads, head_dim), scale, dtype)
