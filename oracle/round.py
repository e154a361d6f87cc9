"""One wavefront round of attention, fp64, two independent formulations.

1. ``round_attention`` -- the mask formulation of "Wave Forcing" Sec. 3.1
   Eq. 4.  Every key token present in round k gets a cleanliness label j
   (live denoising chunk of stage j: j; live store: S; anchor and history:
   S + 1, i.e. cleaner than anything live).  A query token of a task at stage
   s (the store has s = S) sees key token x iff j(x) >= s; the token x token
   mask M[q, x] = 1[j(x) >= s(q)] is materialised and fed to dense softmax
   attention.  This reproduces the contents of Eq. 5: the store sees anchor,
   history and itself (App. B.3), stage s sees anchor, history, store, itself
   and every live j > s; a chunk never sees a later chunk (i' = k - j <= i).

2. ``round_attention_replay`` -- sequential execution (App. B.6,
   Proposition 1): the tasks run one at a time, store first and then stages
   S-1 ... 0; each task first publishes its own K/V (P_{s,l} -> C_{s,l},
   Eq. 8), then attends without any mask over the concatenation of its
   ordered context (Eq. 5), which may only reference K/V already published in
   this round (P_{j,l} -> C_{s,l} for j > s, Eq. 9) or cached by an earlier
   round's store.

K/V of a cached chunk are those its store pass produced (stage S), rotated at
the chunk's own position; the anchor's key is its unrotated store key rotated
at the anchor's position for this round (App. B.3).  Raw per-task Q/K/V come
from a caller-supplied function ``raw(chunk, stage, layer) -> [N_C, 3, H, D]``.

``qk_dtype=Fp8(...)`` models 8-bit attention (the pages' SageAttention
backend, App. B.1 / Sec. 5, with the FP8 K/V pages of App. C.6): Q, K and V
are stored as e4m3 after scaling (saturating at +-448); the anchor's key is
re-rotated from its stored 8-bit unrotated copy once the window has moved.

``qk_dtype="bf16"`` models the pages' BF16 execution (App. B.1: BF16/FA3
reference backend; App. B.2: K/V pages hold the published tensors): Q and K
enter attention as bf16 values after RoPE, so the fp64 rotation is rounded
to bf16 (round-to-nearest-even) before the fp64 attention.  Default None
keeps exact fp64 Q/K.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import schedule as sch
from .attention import masked_attention
from .rope import rope_chunk


@dataclass(frozen=True)
class Fp8:
    """e4m3 storage of Q, K (scaled by qk_scale) and V (scaled by v_scale)."""
    qk_scale: float = 1.0
    v_scale: float = 1.0


def e4m3(x, scale=1.0):
    """Round fp64 values to OCP FP8 e4m3 after multiplying by scale (round
    to nearest even, saturating at +-448 as a satfinite conversion does),
    returned divided by scale again."""
    import torch
    y = np.clip(np.asarray(x, np.float64) * scale, -448.0, 448.0)
    q = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).double().numpy()
    return q / scale


def round_to(x: np.ndarray, qk_dtype):
    """Round fp64 values to the attention input dtype (None: unchanged)."""
    if qk_dtype is None:
        return x
    if isinstance(qk_dtype, Fp8):
        return e4m3(x, qk_dtype.qk_scale)
    if qk_dtype != "bf16":
        raise ValueError(qk_dtype)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def round_v(v: np.ndarray, qk_dtype):
    """V as attention reads it: e4m3 for Fp8 storage, else unchanged (the
    raw values are already in the storage dtype)."""
    if isinstance(qk_dtype, Fp8):
        return e4m3(v, qk_dtype.v_scale)
    return v


@dataclass(frozen=True)
class Geom:
    grid_t: int
    grid_h: int
    grid_w: int
    heads: int
    head_dim: int
    theta: float = 10000.0
    rope_split: tuple | None = None   # (d_t, d_h, d_w); None = the default split

    @property
    def chunk_tokens(self) -> int:
        return self.grid_t * self.grid_h * self.grid_w

    @property
    def grid(self):
        return (self.grid_t, self.grid_h, self.grid_w)


def entry_kv(cfg: sch.Cfg, geom: Geom, e: sch.Entry, layer: int, raw, qk_dtype=None):
    """K (RoPE applied at e.tpos) and V of one context entry: [N_C, H, D] each."""
    producer_stage = e.j if e.kind == sch.KIND_LIVE else cfg.S
    x = np.asarray(raw(e.chunk, producer_stage, layer), dtype=np.float64)
    k_in = x[:, 1]
    if isinstance(qk_dtype, Fp8) and e.kind == sch.KIND_ANCHOR and e.tpos != e.chunk:
        # re-rotated from the stored 8-bit unrotated copy (App. B.3)
        k_in = e4m3(k_in, qk_dtype.qk_scale)
    k = rope_chunk(k_in, e.tpos, geom.grid, geom.theta, geom.rope_split)
    return round_to(k, qk_dtype), round_v(x[:, 2], qk_dtype)


def task_queries(geom: Geom, t: sch.Task, layer: int, raw, qk_dtype=None) -> np.ndarray:
    x = np.asarray(raw(t.chunk, t.stage, layer), dtype=np.float64)
    return round_to(rope_chunk(x[:, 0], t.chunk, geom.grid, geom.theta, geom.rope_split), qk_dtype)


def round_universe(cfg: sch.Cfg, geom: Geom, k: int, layer: int, raw, qk_dtype=None):
    """All key tokens of round k: K, V [H, n_keys, D], labels j, page ids and
    chunk ids [n_keys]."""
    seen = {}
    for t in sch.round_tasks(cfg, k):
        for e in t.context:
            seen[(e.kind, e.chunk, e.j)] = e
    ents = sorted(seen.values(), key=lambda e: (e.kind, e.j, e.chunk))
    ks, vs, lab, pg, ch = [], [], [], [], []
    n = geom.chunk_tokens
    for e in ents:
        kk, vv = entry_kv(cfg, geom, e, layer, raw, qk_dtype)
        ks.append(kk)
        vs.append(vv)
        lab.append(np.full(n, e.j))
        pg.append(np.full(n, e.page))
        ch.append(np.full(n, e.chunk))
    K = np.concatenate(ks, axis=0).transpose(1, 0, 2)
    V = np.concatenate(vs, axis=0).transpose(1, 0, 2)
    return K, V, np.concatenate(lab), np.concatenate(pg), np.concatenate(ch)


def round_attention(cfg: sch.Cfg, geom: Geom, k: int, layer: int, raw,
                    rows=None, universe=None, qk_dtype=None):
    """Mask formulation.  Returns one array [n_rows, H, D] per task (slot order).

    ``rows`` (optional) selects query rows of every task (same indices for all
    tasks); each output row depends on its own query row only."""
    K, V, lab, _, _ = (universe if universe is not None
                       else round_universe(cfg, geom, k, layer, raw, qk_dtype))
    outs = []
    for t in sch.round_tasks(cfg, k):
        q = task_queries(geom, t, layer, raw, qk_dtype)
        if rows is not None:
            q = q[np.asarray(rows)]
        mask = np.broadcast_to(sch.sees(cfg, t.stage, lab)[None, :], (q.shape[0], lab.shape[0]))
        o = masked_attention(q.transpose(1, 0, 2), K, V, mask)
        outs.append(o.transpose(1, 0, 2))
    return outs


def round_attention_replay(cfg: sch.Cfg, geom: Geom, k: int, layer: int, raw):
    """Sequential replay (store, then stages S-1 .. 0) over ordered contexts,
    unmasked.  Returns one array [N_C, H, D] per task in slot order."""
    tasks = sch.round_tasks(cfg, k)
    published = {}
    outs = {}
    for t in sorted(tasks, key=lambda t: -t.stage):
        own = sch.Entry(sch.KIND_STORE if t.stage == cfg.S else sch.KIND_LIVE,
                        t.chunk, t.stage, t.dest_page, t.chunk)
        published[(t.chunk, t.stage)] = entry_kv(cfg, geom, own, layer, raw)
        ks, vs = [], []
        for e in t.context:
            if e.kind in (sch.KIND_STORE, sch.KIND_LIVE):
                key = (e.chunk, e.j)
                if key not in published:
                    raise AssertionError(f"task {t.chunk, t.stage} reads unpublished {key}")
                kk, vv = published[key]
            else:
                kk, vv = entry_kv(cfg, geom, e, layer, raw)
            ks.append(kk)
            vs.append(vv)
        K = np.concatenate(ks, axis=0).transpose(1, 0, 2)
        V = np.concatenate(vs, axis=0).transpose(1, 0, 2)
        q = task_queries(geom, t, layer, raw)
        mask = np.ones((q.shape[0], K.shape[1]), dtype=bool)
        outs[(t.chunk, t.stage)] = masked_attention(q.transpose(1, 0, 2), K, V, mask).transpose(1, 0, 2)
    return [outs[(t.chunk, t.stage)] for t in tasks]


def round_flops(cfg: sch.Cfg, geom: Geom, k: int) -> int:
    """Algorithmic attention FLOPs of round k: 4 * N_C * keys * D per task and head."""
    n = geom.chunk_tokens
    return sum(4 * n * sch.key_count(t, n) * geom.head_dim * geom.heads
               for t in sch.round_tasks(cfg, k))
