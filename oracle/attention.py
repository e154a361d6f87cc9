"""Dense masked softmax attention in fp64 (the textbook definition).

O = softmax(Q K^T * scale + log M) V, per head, with M a materialised boolean
mask; a masked entry contributes exactly 0 and the softmax subtracts the row
maximum first.  The scale is 1/sqrt(head_dim) (the pages are silent; the
standard choice).
"""

from __future__ import annotations

import numpy as np


def masked_softmax(scores: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Row softmax of ``scores`` [..., n_q, n_k] restricted to ``mask`` (bool,
    broadcastable).  Every row must have at least one visible key."""
    s = np.where(mask, scores, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.where(mask, np.exp(s - m), 0.0)
    return e / e.sum(axis=-1, keepdims=True)


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     mask: np.ndarray, scale: float | None = None) -> np.ndarray:
    """q [H, n_q, D], k/v [H, n_k, D], mask [n_q, n_k] -> O [H, n_q, D] (fp64)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    scores = np.matmul(q, np.swapaxes(k, -1, -2)) * scale
    p = masked_softmax(scores, mask[None, :, :])
    return np.matmul(p, v)
