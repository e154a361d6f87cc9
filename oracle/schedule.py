"""Wavefront schedule, cache pages and ordered contexts (fp-free, integer).

Written from "Wave Forcing: Towards Speed-of-Light Streaming Video
Generation":

* Sec. 2 Eq. 2 -- the wavefront state set F_k plus the store B_{k-S}; width
  at most S+1.
* Sec. 3.1 Eq. 3 -- cell (i, s) runs in round k = i + s; store at (k-S, S);
  active set A_k = {s : 0 <= s < S, 0 <= k-s < N_chunk}; store active iff
  0 <= k-S < N_chunk.
* Sec. 3.1 Eq. 5 -- ordered context: anchor, bounded clean history, live
  store, then denoising K/V in increasing stage j >= s (self first).
* App. B.3 (Algorithm 1 and "Round schedule and cache semantics") --
  N_chunk + S rounds; the live store page becomes history after the round;
  the first clean chunk is a persistent anchor whose unrotated key is kept so
  RoPE can be re-applied when the window shifts; the store attends to anchor,
  retained history and itself.
* App. B.4 Eq. 16 -- slot occupancy eta = N_chunk / (N_chunk + S).
* App. B.8 -- fixed page capacity: anchor, bounded history, live store and at
  most S denoising chunks.

Two comparison graphs the pages define next to WF, on the same pages:

* RF mask (Sec. 3.1, the reverse refinement of Rolling Forcing that Eq. 4
  removes; Sec. 5.5 "RF's full active-window attention"): a denoising task
  also reads the noisier live chunks of the window, M_RF(s, j) = 1 for all
  s, j in A_k.  The store keeps the WF store context (reading: the reverse
  edges are between denoising slots).
* Sequential schedule (Sec. 2, NF1C): chunk after chunk, its S denoising
  forwards and then its store pass, one task per round; round r runs chunk
  r // (S+1) at stage r % (S+1), attending to anchor, history and itself.

Readings where the pages are silent (each also listed in the design notes):

* W ("history_chunks") counts clean history chunks *excluding* the anchor and
  the live store; -1 keeps every clean chunk.  History is ordered oldest first.
* Before chunk 0 is stored there is no anchor; the store pass of chunk 0
  writes the anchor page itself and attends only to itself.
* Anchor position (mode ADJACENT, default): the anchor's temporal chunk
  position is one before the oldest non-anchor chunk present in the round
  (history, store or live), clamped at 0; with full history it never moves.
  Mode ABSOLUTE keeps it at chunk position 0.
* The store's longer prefix (App. B.3: under a token budget the store
  reserves one query chunk where a denoising task reserves S, so their
  prefixes can differ): by default both use the same W history chunks; the
  option store_extra = E >= 0 (with bounded history) lets the store keep the
  E next-older clean chunks too.  E = S gives the store the key count of a
  stage-0 denoising task (anchor + W + store + S live = anchor + W + S +
  itself).
* Page ids are this implementation's own convention, written here in closed
  form so the library's ring allocator can be checked against it bit for bit:
  page 0 = anchor; ring pages 1..R hold clean chunks, chunk c on page
  1 + ((c - c0) mod R) with c0 = 1 (anchor on) or 0; R = W + E + 1 (the
  store's history + the live store), or every non-anchor chunk for full
  history; the live denoising chunk of stage s is on page 1 + R + s; page
  1 + R + S keeps the anchor's unrotated key.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

ANCHOR_ADJACENT = 0
ANCHOR_ABSOLUTE = 1

MASK_WF = 0
MASK_RF = 1

# cleanliness labels j of Eq. 4, extended to the cached entries of Eq. 5
# (anchor and history S+1, live store S, the store's extra history S+2)
KIND_ANCHOR = 0
KIND_HISTORY = 1
KIND_STORE = 2
KIND_LIVE = 3


@dataclass(frozen=True)
class Cfg:
    S: int                 # denoising steps; the store is stage S
    n_chunks: int          # N_chunk
    history: int           # W, -1 = keep all clean chunks
    use_anchor: bool = True
    anchor_mode: int = ANCHOR_ADJACENT
    mask: int = MASK_WF
    sequential: bool = False
    store_extra: int = 0   # E: extra history chunks of the store (bounded history only)


@dataclass(frozen=True)
class Entry:
    """One segment of an ordered context (one chunk's K/V)."""
    kind: int      # KIND_*
    chunk: int     # chunk index i
    j: int         # cleanliness label: live stage j, S for the store, S+1 for anchor/history
    page: int      # page id (closed form above)
    tpos: int      # temporal chunk position its keys are rotated at


@dataclass(frozen=True)
class Task:
    chunk: int
    stage: int     # s < S denoising, s == S store
    dest_page: int # page its K/V are published to
    context: tuple # tuple[Entry, ...] in Eq. 5 order


def n_rounds(cfg: Cfg) -> int:
    """Algorithm 1 runs rounds k = 0 .. N_chunk + S - 1 (App. B.3); the
    sequential schedule runs N_chunk (S+1) single-task rounds."""
    if cfg.sequential:
        return cfg.n_chunks * (cfg.S + 1)
    return cfg.n_chunks + cfg.S


def live_tasks(cfg: Cfg, k: int) -> list[tuple[int, int]]:
    """(chunk, stage) of the denoising tasks of round k, stages ascending:
    A_k of Sec. 3.1 (after Eq. 3) with chunk k - s, or the one task of a
    sequential round."""
    if cfg.sequential:
        i, s = divmod(k, cfg.S + 1)
        return [(i, s)] if s < cfg.S else []
    return [(k - s, s) for s in range(cfg.S) if 0 <= k - s < cfg.n_chunks]


def active_stages(cfg: Cfg, k: int) -> list[int]:
    """A_k of Sec. 3.1 (after Eq. 3)."""
    return [s for _, s in live_tasks(cfg, k)]


def store_chunk(cfg: Cfg, k: int):
    """Chunk refreshed by the store at round k, or None (Sec. 3.1)."""
    if cfg.sequential:
        i, s = divmod(k, cfg.S + 1)
        return i if s == cfg.S else None
    u = k - cfg.S
    return u if 0 <= u < cfg.n_chunks else None


def sees(cfg: Cfg, s: int, j):
    """Mask of Sec. 3.1 Eq. 4 extended to the labels of cached entries
    (anchor/history S+1, live store S): WF 1[j >= s]; RF lets a denoising
    query see every live label of the window as well.  History kept for the
    store only (store_extra > 0) carries label S+2, which only the store
    (s = S) sees -- no label of Eq. 4's form j >= s can express that."""
    if cfg.mask == MASK_RF and s < cfg.S:
        base = j >= 0                      # every label (elementwise for arrays)
    else:
        base = j >= s
    if cfg.store_extra > 0 and s < cfg.S:
        return np.logical_and(base, np.asarray(j) != cfg.S + 2)
    return base


def ring_size(cfg: Cfg) -> int:
    if cfg.history >= 0:
        return cfg.history + cfg.store_extra + 1
    return max(1, cfg.n_chunks - (1 if cfg.use_anchor else 0))


def n_pages(cfg: Cfg) -> int:
    return 1 + ring_size(cfg) + cfg.S + 1


def clean_page(cfg: Cfg, c: int) -> int:
    if cfg.use_anchor and c == 0:
        return 0
    c0 = 1 if cfg.use_anchor else 0
    return 1 + (c - c0) % ring_size(cfg)


def live_page(cfg: Cfg, s: int) -> int:
    return 1 + ring_size(cfg) + s


def raw_anchor_page(cfg: Cfg) -> int:
    return 1 + ring_size(cfg) + cfg.S


def clean_before(cfg: Cfg, k: int) -> list[int]:
    """Chunks whose store finished in an earlier round: c + S < k (the
    store of chunk c runs in round c + S; round c (S+1) + S sequentially)."""
    if cfg.sequential:
        return [c for c in range(cfg.n_chunks) if c * (cfg.S + 1) + cfg.S < k]
    return [c for c in range(cfg.n_chunks) if c + cfg.S < k]


def anchor_present(cfg: Cfg, k: int) -> bool:
    return cfg.use_anchor and 0 in clean_before(cfg, k)


def history_chunks(cfg: Cfg, k: int, store: bool = False) -> list[int]:
    """Bounded clean history H_k: the W newest clean non-anchor chunks, oldest
    first; the store's keeps the W + E newest."""
    clean = [c for c in clean_before(cfg, k) if not (cfg.use_anchor and c == 0)]
    if cfg.history >= 0:
        keep = cfg.history + (cfg.store_extra if store else 0)
        clean = clean[max(0, len(clean) - keep):] if keep > 0 else []
    return clean


def anchor_tpos(cfg: Cfg, k: int) -> int:
    """Temporal chunk position the anchor's key is rotated at in round k."""
    if cfg.anchor_mode == ANCHOR_ABSOLUTE:
        return 0
    others = list(history_chunks(cfg, k, store=True))
    u = store_chunk(cfg, k)
    if u is not None and not (cfg.use_anchor and u == 0):
        others.append(u)
    others += [c for c, _ in live_tasks(cfg, k)]
    if not others:
        return 0
    return max(0, min(others) - 1)


def round_tasks(cfg: Cfg, k: int) -> list[Task]:
    """The tasks of round k in slot order (stages ascending, then the store),
    each with its ordered context (Eq. 5; store context per App. B.3)."""
    S = cfg.S
    live = live_tasks(cfg, k)
    u = store_chunk(cfg, k)
    anchor = []
    if anchor_present(cfg, k):
        anchor.append(Entry(KIND_ANCHOR, 0, S + 1, 0, anchor_tpos(cfg, k)))
    prefix = anchor + [Entry(KIND_HISTORY, h, S + 1, clean_page(cfg, h), h)
                       for h in history_chunks(cfg, k)]
    window = set(history_chunks(cfg, k))
    store_prefix = anchor + [Entry(KIND_HISTORY, h, S + 1 if h in window else S + 2, clean_page(cfg, h), h)
                             for h in history_chunks(cfg, k, store=True)]
    store_entry = None
    if u is not None:
        store_entry = Entry(KIND_STORE, u, S, clean_page(cfg, u), u)
    tasks = []
    for c, s in live:
        ctx = list(prefix)
        if store_entry is not None:
            ctx.append(store_entry)
        for c2, j in live:
            if sees(cfg, s, j):
                ctx.append(Entry(KIND_LIVE, c2, j, live_page(cfg, j), c2))
        tasks.append(Task(c, s, live_page(cfg, s), tuple(ctx)))
    if u is not None:
        ctx = list(store_prefix) + [store_entry]
        tasks.append(Task(u, S, clean_page(cfg, u), tuple(ctx)))
    return tasks


def slot_occupancy(cfg: Cfg) -> float:
    """eta_slot = N_chunk / (N_chunk + S) (App. B.4 Eq. 16); a sequential
    schedule keeps one of the S+1 slots busy per round."""
    if cfg.sequential:
        return 1.0 / (cfg.S + 1)
    return cfg.n_chunks / (cfg.n_chunks + cfg.S)


def key_count(task: Task, chunk_tokens: int) -> int:
    return len(task.context) * chunk_tokens
