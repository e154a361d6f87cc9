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


def dit_params(seed: int, dim: int, ffn: int, layers: int, channels: int = 16,
               freq: int = 256, std: float = 0.02, dtype=torch.bfloat16,
               norm_gain: float = 1.0) -> dict:
    """Random-initialised DiT parameters ~ N(0, std^2), rounded to ``dtype``.

    Matrices are [out, in] (the layout of a linear layer's weight).  Keys:
    patch_w [dim, 4C], patch_b, t1_w [dim, freq], t1_b, t2_w [dim, dim],
    t2_b, tp_w [6 dim, dim], tp_b, head_w [4C, dim], head_b, head_mod
    [2, dim]; per layer (lists of length ``layers``): qkv_w [3 dim, dim],
    qkv_b, o_w [dim, dim], o_b, f1_w [ffn, dim], f1_b, f2_w [dim, ffn], f2_b,
    mod [6, dim], and the q / k RMSNorm gains nq, nk [dim] drawn as
    ``norm_gain`` + N(0, std^2) (a normalisation gain starts at 1; the draw
    makes every channel's gain distinct)."""
    p = 4 * channels

    def g(tag, *shape):
        return normal(key_of(seed, 7, *tag), shape, std, dtype)

    out = {
        "patch_w": g((0, 0), dim, p), "patch_b": g((0, 1), dim),
        "t1_w": g((1, 0), dim, freq), "t1_b": g((1, 1), dim),
        "t2_w": g((2, 0), dim, dim), "t2_b": g((2, 1), dim),
        "tp_w": g((3, 0), 6 * dim, dim), "tp_b": g((3, 1), 6 * dim),
        "head_w": g((4, 0), p, dim), "head_b": g((4, 1), p),
        "head_mod": g((4, 2), 2, dim),
    }
    per = {"qkv_w": (3 * dim, dim), "qkv_b": (3 * dim,), "o_w": (dim, dim), "o_b": (dim,),
           "f1_w": (ffn, dim), "f1_b": (ffn,), "f2_w": (dim, ffn), "f2_b": (dim,),
           "mod": (6, dim)}
    for i, (name, shape) in enumerate(per.items()):
        out[name] = [g((10, l, i), *shape) for l in range(layers)]
    for i, name in ((9, "nq"), (10, "nk")):
        out[name] = [(norm_gain + normal(key_of(seed, 7, 10, l, i), (dim,), std)).to(dtype)
                     for l in range(layers)]
    return out


def latent(seed: int, chunk: int, stage: int, channels: int, frames: int, height: int,
           width: int) -> torch.Tensor:
    """N(0, 1) fp32 latent draw keyed by (chunk, stage): [C, F, H, W].  Used
    both as the fresh noise of a chunk (stage -1) and as the transition draw
    eps_{chunk, stage}."""
    return normal(key_of(seed, 2, chunk, stage), (channels, frames, height, width), 1.0,
                  torch.float32)
