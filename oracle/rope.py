"""3D rotary position embedding in fp64.

The paper applies RoPE to Q and K right after the QKV projection and before
K/V are published ("Wave Forcing", Sec. 4.2; App. B.3 keeps the anchor's
unrotated key so RoPE can be re-applied).  It does not print the axis split,
the base or the pair convention, so this oracle adopts the Wan2.1 video
convention as its reading (stated again in the design notes):

* head_dim D is split into a temporal, a height and a width part of sizes
  D - 4*floor(D/6), 2*floor(D/6), 2*floor(D/6)  (128 -> 44/42/42), unless a
  split (d_t, d_h, d_w) of even sizes summing to D is given (a plan option);
* channels are rotated in interleaved pairs (2m, 2m+1);
* pair m of a part of size d rotates by angle pos * theta^(-2m/d), theta = 1e4;
* (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a);
* a token's position is (t, h, w) with t the absolute latent frame
  (grid_t * chunk_position + frame) and (h, w) its patch-grid cell; tokens of
  a chunk are ordered frame-major, then h, then w.

Parity of the convention is internal (unpinned against the paper); the
rotation itself is pinned by norm preservation, relative-position invariance,
composition and closed-form special cases in the tests.
"""

from __future__ import annotations

import numpy as np


def sections(head_dim: int, split=None) -> tuple[int, int, int]:
    """Sizes of the (t, h, w) parts of the head dimension."""
    if split is not None:
        dt, dh, dw = (int(v) for v in split)
        if min(dt, dh, dw) < 0 or dt % 2 or dh % 2 or dw % 2 or dt + dh + dw != head_dim:
            raise ValueError(f"bad RoPE split {split} for head_dim {head_dim}")
        return dt, dh, dw
    q = head_dim // 6
    return head_dim - 4 * q, 2 * q, 2 * q


def pair_angles(head_dim: int, theta: float, t, h, w, split=None) -> np.ndarray:
    """Angles [n, head_dim/2] for positions given as arrays t, h, w of length n."""
    dt, dh, dw = sections(head_dim, split)
    t = np.asarray(t, dtype=np.float64)[:, None]
    h = np.asarray(h, dtype=np.float64)[:, None]
    w = np.asarray(w, dtype=np.float64)[:, None]
    parts = []
    for pos, d in ((t, dt), (h, dh), (w, dw)):
        m = np.arange(d // 2, dtype=np.float64)
        inv_freq = theta ** (-2.0 * m / d)
        parts.append(pos * inv_freq[None, :])
    return np.concatenate(parts, axis=1)


def rotate(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate interleaved pairs of x [n, ..., D] by angles [n, D/2] (fp64).

    Extra middle axes (e.g. heads) share the token's angles."""
    x = np.asarray(x, dtype=np.float64)
    a = angles.reshape(angles.shape[0], *([1] * (x.ndim - 2)), angles.shape[1])
    c, s = np.cos(a), np.sin(a)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def chunk_positions(chunk_tpos: int, grid_t: int, grid_h: int, grid_w: int):
    """(t, h, w) of every token of a chunk placed at temporal chunk position
    ``chunk_tpos``; tokens are frame-major, then h, then w."""
    n = np.arange(grid_t * grid_h * grid_w)
    f = n // (grid_h * grid_w)
    hh = (n // grid_w) % grid_h
    ww = n % grid_w
    return grid_t * chunk_tpos + f, hh, ww


def rope_chunk(x: np.ndarray, chunk_tpos: int, grid, theta: float, split=None) -> np.ndarray:
    """RoPE for a whole chunk x [N_C, H, D] placed at ``chunk_tpos``."""
    t, h, w = chunk_positions(chunk_tpos, *grid)
    return rotate(x, pair_angles(x.shape[-1], theta, t, h, w, split))
