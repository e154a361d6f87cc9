"""Pins of the oracle's schedule against what the paper fixes.

"Wave Forcing" Sec. 2 Eq. 2 (width <= S+1, N = S+1 forwards per chunk),
Sec. 3.1 Eq. 3-5, Sec. 4.2 Eq. 10, App. B.3 (N_chunk + S rounds, store
context), App. B.4 Eq. 16 (eta = 133/137 = 97.1% at S=4).
"""

import itertools

import pytest

from oracle import schedule as sch
from golden_io import read_schedule


def _as_tuples(tasks):
    return [(t.chunk, t.stage, t.dest_page,
             [(e.kind, e.chunk, e.j, e.page, e.tpos) for e in t.context]) for t in tasks]


@pytest.mark.parametrize("name,cfg", [
    ("schedule_s2_n6_full.txt", sch.Cfg(S=2, n_chunks=6, history=-1)),
    ("schedule_s4_n10_w3.txt", sch.Cfg(S=4, n_chunks=10, history=3)),
])
def test_hand_worked_rounds(name, cfg):
    gold = read_schedule(name)
    for k, tasks in gold.items():
        assert _as_tuples(sch.round_tasks(cfg, k)) == tasks, f"round {k}"
    if name.startswith("schedule_s2"):
        assert sorted(gold) == list(range(sch.n_rounds(cfg)))


CFGS = [sch.Cfg(S, N, W, anchor, mode)
        for S, N, W, anchor, mode in itertools.product(
            [1, 2, 3, 4, 5], [1, 2, 3, 6, 11], [-1, 0, 1, 3], [True, False],
            [sch.ANCHOR_ADJACENT, sch.ANCHOR_ABSOLUTE])]


@pytest.mark.parametrize("cfg", CFGS, ids=str)
def test_schedule_invariants(cfg):
    S, N = cfg.S, cfg.n_chunks
    seen = {}
    stores = []
    for k in range(-2, sch.n_rounds(cfg) + 3):
        tasks = sch.round_tasks(cfg, k)
        if k < 0 or k >= sch.n_rounds(cfg):
            assert tasks == []          # Algorithm 1 runs k = 0 .. N+S-1 only
            continue
        assert 1 <= len(tasks) <= S + 1          # Eq. 2 width
        for t in tasks:
            # Eq. 3: cell (i, s) runs in round k = i + s; store at (k-S, S)
            assert t.chunk + t.stage == k
            assert 0 <= t.chunk < N
            seen.setdefault(t.chunk, []).append(t.stage)
            # self first among live entries; the task reads its own K/V
            own = [e for e in t.context if e.chunk == t.chunk and e.j == t.stage]
            assert len(own) == 1 and own[0].page == t.dest_page
            # a chunk never sees a later chunk (Sec. 3.1 after Eq. 4)
            assert all(e.chunk <= t.chunk for e in t.context)
            # Eq. 5 ordering: anchor, history (oldest first), store, live j ascending
            kinds = [e.kind for e in t.context]
            assert kinds == sorted(kinds)
            hist = [e.chunk for e in t.context if e.kind == sch.KIND_HISTORY]
            assert hist == sorted(hist)
            live = [e.j for e in t.context if e.kind == sch.KIND_LIVE]
            assert live == sorted(live) and all(j >= t.stage for j in live)
            if t.stage == S:
                # store attends to anchor, retained history and itself (App. B.3)
                assert all(e.kind != sch.KIND_LIVE for e in t.context)
            # bounded window keeps the W newest clean non-anchor chunks, or all
            # of them while fewer than W exist (App. B.3, Sec. 3.1 Eq. 5)
            clean = [c for c in range(N) if c + S < k and not (cfg.use_anchor and c == 0)]
            want = clean if cfg.history < 0 else clean[len(clean) - min(len(clean), cfg.history):]
            assert hist == want
            # pages of one context are distinct (fixed slots, App. B.2 Eq. 13)
            pages = [e.page for e in t.context]
            assert len(set(pages)) == len(pages)
            assert all(0 <= p < sch.n_pages(cfg) - 1 for p in pages)
        store = [t for t in tasks if t.stage == S]
        stores.append(store[0].chunk if store else None)
    # every chunk gets exactly S denoising updates plus one store: N = S+1 forwards
    assert sorted(seen) == list(range(N))
    assert all(sorted(v) == list(range(S + 1)) for v in seen.values())
    # after fill, exactly one completed chunk per round, in order
    assert stores[:S] == [None] * S
    assert stores[S:] == list(range(N))
    # all S+1 slots busy only for S <= k < N (App. B.4); never if N <= S
    full = [k for k in range(sch.n_rounds(cfg)) if len(sch.round_tasks(cfg, k)) == S + 1]
    assert full == list(range(S, N))


def test_slot_occupancy_printed_example():
    # App. B.4: "133/137 = 97.1%" for 399 latent frames (133 chunks) at S=4
    cfg = sch.Cfg(S=4, n_chunks=133, history=3)
    eta = sch.slot_occupancy(cfg)
    assert (cfg.n_chunks, cfg.n_chunks + cfg.S) == (133, 137)
    assert round(100 * eta, 1) == 97.1
    busy = sum(len(sch.round_tasks(cfg, k)) for k in range(sch.n_rounds(cfg)))
    assert busy == 133 * 5                 # N_chunk (S+1) forwards in all
    assert busy / (sch.n_rounds(cfg) * (cfg.S + 1)) == pytest.approx(eta)


@pytest.mark.parametrize("S,W", [(4, 3), (5, 3), (2, 1), (3, 0)])
def test_key_counts_eq10(S, W):
    # Sec. 4.2 Eq. 10: N_s = N_prefix + (S - s) N_C in a filled round, with
    # N_prefix covering anchor + history + store.
    cfg = sch.Cfg(S=S, n_chunks=40, history=W)
    nc = 7
    k = S + W + 5
    tasks = sch.round_tasks(cfg, k)
    prefix = (1 + W + 1) * nc
    for t in tasks:
        if t.stage < S:
            assert sch.key_count(t, nc) == prefix + (S - t.stage) * nc
        else:
            assert sch.key_count(t, nc) == prefix


def test_anchor_positions():
    cfg = sch.Cfg(S=4, n_chunks=20, history=3)
    # anchor sits one chunk before the oldest non-anchor chunk of the round
    for k in range(sch.n_rounds(cfg)):
        if not sch.anchor_present(cfg, k):
            continue
        hist = sch.history_chunks(cfg, k)
        assert sch.anchor_tpos(cfg, k) == max(0, (hist[0] if hist else 1) - 1)
    absolute = sch.Cfg(S=4, n_chunks=20, history=3, anchor_mode=sch.ANCHOR_ABSOLUTE)
    assert all(sch.anchor_tpos(absolute, k) == 0 for k in range(sch.n_rounds(absolute)))
    full = sch.Cfg(S=4, n_chunks=20, history=-1)
    assert all(sch.anchor_tpos(full, k) == 0 for k in range(sch.n_rounds(full)))


def test_planted_mistake_is_caught(monkeypatch):
    """A store that also read live chunks (a plausible slip) breaks the golden rounds."""
    real = sch.round_tasks

    def wrong(cfg, k):
        out = []
        for t in real(cfg, k):
            if t.stage == cfg.S:
                live = [e for t2 in real(cfg, k) for e in t2.context if e.kind == sch.KIND_LIVE]
                t = sch.Task(t.chunk, t.stage, t.dest_page, t.context + tuple(live[:1]))
            out.append(t)
        return out

    monkeypatch.setattr(sch, "round_tasks", wrong)
    gold = read_schedule("schedule_s2_n6_full.txt")
    cfg = sch.Cfg(S=2, n_chunks=6, history=-1)
    assert any(_as_tuples(sch.round_tasks(cfg, k)) != v for k, v in gold.items())


# ---- comparison graphs: RF mask and the sequential (NF1C) schedule -----------

def _tuples(tasks):
    return [(t.chunk, t.stage, t.dest_page,
             tuple((e.kind, e.chunk, e.j, e.page, e.tpos) for e in t.context)) for t in tasks]


@pytest.mark.parametrize("S,N,W", [(4, 12, 3), (2, 6, -1), (3, 7, 1)])
def test_rf_mask_adds_exactly_the_reverse_edges(S, N, W):
    """RF (Sec. 3.1: the reverse refinement Eq. 4 removes; Sec. 5.5 'full
    active-window attention'): a denoising task additionally reads the live
    chunks of noisier stages j < s, i.e. later chunks i' = k - j > i; nothing
    else changes (pages, store context, prefix)."""
    wf_cfg = sch.Cfg(S=S, n_chunks=N, history=W)
    rf_cfg = sch.Cfg(S=S, n_chunks=N, history=W, mask=sch.MASK_RF)
    for k in range(sch.n_rounds(wf_cfg)):
        a, b = sch.round_tasks(wf_cfg, k), sch.round_tasks(rf_cfg, k)
        assert [(t.chunk, t.stage, t.dest_page) for t in a] == [(t.chunk, t.stage, t.dest_page) for t in b]
        live = [(t.chunk, t.stage) for t in a if t.stage < S]
        for ta, tb in zip(a, b):
            if ta.stage == S:
                assert ta.context == tb.context
                continue
            extra = [e for e in tb.context if e not in ta.context]
            assert all(e in tb.context for e in ta.context)
            assert sorted((e.chunk, e.j) for e in extra) == sorted((c, s) for c, s in live if s < ta.stage)
            assert all(e.kind == sch.KIND_LIVE and e.chunk > ta.chunk for e in extra)
            assert sch.key_count(tb, 7) == sch.key_count(ta, 7) + 7 * len(extra)


def test_rf_has_no_sequential_order():
    """With reverse edges a cleaner task reads a noisier task of the same
    round and vice versa, so no task-at-a-time order exists (the dependency
    cycle Wave Parallelism needs removed, Sec. 4.1); WF replays in order."""
    from oracle.round import Geom, round_attention_replay
    import numpy as np
    geom = Geom(1, 2, 2, 1, 8)
    raw = lambda c, s, l: np.ones((4, 3, 1, 8))
    k = 3
    round_attention_replay(sch.Cfg(S=3, n_chunks=6, history=1), geom, k, 0, raw)
    with pytest.raises(AssertionError):
        round_attention_replay(sch.Cfg(S=3, n_chunks=6, history=1, mask=sch.MASK_RF), geom, k, 0, raw)


def test_sequential_schedule_hand_worked():
    """NF1C (Sec. 2): chunk after chunk, S denoising forwards then the store,
    one task per round, each attending to anchor, history and itself.
    S = 2, N = 3, W = 1: ring of R = 2 pages (1, 2), live pages 3 + s, anchor
    page 0 (derived by hand from Eq. 5 and App. B.3)."""
    cfg = sch.Cfg(S=2, n_chunks=3, history=1, sequential=True)
    A, H, U, L = sch.KIND_ANCHOR, sch.KIND_HISTORY, sch.KIND_STORE, sch.KIND_LIVE
    want = {
        0: [(0, 0, 3, ((L, 0, 0, 3, 0),))],
        1: [(0, 1, 4, ((L, 0, 1, 4, 0),))],
        2: [(0, 2, 0, ((U, 0, 2, 0, 0),))],
        3: [(1, 0, 3, ((A, 0, 3, 0, 0), (L, 1, 0, 3, 1)))],
        4: [(1, 1, 4, ((A, 0, 3, 0, 0), (L, 1, 1, 4, 1)))],
        5: [(1, 2, 1, ((A, 0, 3, 0, 0), (U, 1, 2, 1, 1)))],
        6: [(2, 0, 3, ((A, 0, 3, 0, 0), (H, 1, 3, 1, 1), (L, 2, 0, 3, 2)))],
        7: [(2, 1, 4, ((A, 0, 3, 0, 0), (H, 1, 3, 1, 1), (L, 2, 1, 4, 2)))],
        8: [(2, 2, 2, ((A, 0, 3, 0, 0), (H, 1, 3, 1, 1), (U, 2, 2, 2, 2)))],
    }
    assert sch.n_rounds(cfg) == 9
    for k, v in want.items():
        assert _tuples(sch.round_tasks(cfg, k)) == v, k


@pytest.mark.parametrize("S,N,W", [(4, 9, 3), (2, 5, -1), (3, 4, 0), (1, 3, 1)])
def test_sequential_schedule_invariants(S, N, W):
    cfg = sch.Cfg(S=S, n_chunks=N, history=W, sequential=True)
    seen = []
    for k in range(sch.n_rounds(cfg)):
        tasks = sch.round_tasks(cfg, k)
        assert len(tasks) == 1                       # one forward per round
        t = tasks[0]
        seen.append((t.chunk, t.stage))
        assert (t.chunk, t.stage) == divmod(k, S + 1)
        own = [e for e in t.context if e.kind in (sch.KIND_LIVE, sch.KIND_STORE)]
        assert [(e.chunk, e.j) for e in own] == [(t.chunk, t.stage)]
        hist = [e.chunk for e in t.context if e.kind == sch.KIND_HISTORY]
        clean = list(range(1, t.chunk))
        assert hist == (clean if W < 0 else clean[len(clean) - min(len(clean), W):])
        assert any(e.kind == sch.KIND_ANCHOR for e in t.context) == (t.chunk > 0)
    # N = S + 1 forwards per chunk (NF1C), chunks strictly in order
    assert seen == [(i, s) for i in range(N) for s in range(S + 1)]
    assert sch.slot_occupancy(cfg) == pytest.approx(1 / (S + 1))


# ---- the store's longer prefix (App. B.3: the store reserves one query chunk,
# a denoising task S, so under a token budget the store may keep more history)

EXTRA = [sch.Cfg(4, 14, 3, store_extra=4), sch.Cfg(2, 9, 0, store_extra=2),
         sch.Cfg(3, 10, 1, store_extra=1, use_anchor=False),
         sch.Cfg(3, 10, 2, store_extra=3, mask=sch.MASK_RF),
         sch.Cfg(2, 5, 1, store_extra=2, sequential=True),
         sch.Cfg(3, 9, 2, store_extra=3, anchor_mode=sch.ANCHOR_ABSOLUTE)]


@pytest.mark.parametrize("cfg", EXTRA, ids=str)
def test_store_extra_history_contexts(cfg):
    """Denoising tasks keep the W newest clean chunks, the store the W + E
    newest (label S + 2 on the ones only it keeps); within a round no page
    holds two chunks; the adjacent anchor sits before the oldest kept chunk."""
    W, E, S = cfg.history, cfg.store_extra, cfg.S
    for k in range(sch.n_rounds(cfg)):
        clean = [c for c in sch.clean_before(cfg, k) if not (cfg.use_anchor and c == 0)]
        page_of = {}
        for t in sch.round_tasks(cfg, k):
            hist = [e for e in t.context if e.kind == sch.KIND_HISTORY]
            keep = W + E if t.stage == S else W
            assert [e.chunk for e in hist] == clean[max(0, len(clean) - keep):] if keep else hist == []
            for e in hist:
                only_store = e.chunk not in clean[max(0, len(clean) - W):] if W else True
                assert e.j == (S + 2 if only_store else S + 1)
                assert t.stage == S or not only_store
            for e in t.context:
                if e.kind != sch.KIND_LIVE:
                    assert page_of.setdefault(e.page, e.chunk) == e.chunk, (k, e)
        if sch.anchor_present(cfg, k) and cfg.anchor_mode == sch.ANCHOR_ADJACENT:
            store_hist = sch.history_chunks(cfg, k, store=True)
            if store_hist:
                assert sch.anchor_tpos(cfg, k) == store_hist[0] - 1


def test_store_extra_equal_to_s_equalises_the_key_budget():
    """With E = S the store reads as many key chunks as a stage-0 task once
    the history is full (anchor + W + E + itself = anchor + W + store + S)."""
    for S, W in ((2, 1), (4, 3), (3, 0)):
        cfg = sch.Cfg(S, 20, W, store_extra=S)
        seen = 0
        for k in range(sch.n_rounds(cfg)):
            tasks = sch.round_tasks(cfg, k)
            clean = [c for c in sch.clean_before(cfg, k) if c != 0]
            if len(tasks) == S + 1 and len(clean) >= W + S:
                assert len(tasks[-1].context) == len(tasks[0].context) == 1 + W + S + 1
                seen += 1
        assert seen > 0


def test_store_extra_zero_is_the_default_schedule():
    for cfg in (sch.Cfg(4, 12, 3), sch.Cfg(2, 6, -1), sch.Cfg(3, 7, 1, mask=sch.MASK_RF)):
        alt = sch.Cfg(cfg.S, cfg.n_chunks, cfg.history, cfg.use_anchor, cfg.anchor_mode, cfg.mask,
                      cfg.sequential, store_extra=0)
        for k in range(sch.n_rounds(cfg)):
            assert sch.round_tasks(cfg, k) == sch.round_tasks(alt, k)
