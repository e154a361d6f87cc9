"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every symbol include/wf.h declares, argument validation returns the
documented codes, and the library's schedule / page ring matches the oracle
bit for bit ("Wave Forcing" Sec. 3.1 Eq. 3-5, App. B.3)."""

import ctypes
import itertools
import os
import re

import pytest

import chunk_causal_dit_round_b300 as wf
from oracle import schedule as sch

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "wf.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wf_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_are_exported():
    names = declared_functions()
    assert len(names) >= 10
    assert sorted(names) == sorted(wf.SYMBOLS)
    for n in names:
        assert hasattr(wf.lib, n), n


def _plan(S, NC, H, D, W, **kw):
    o = wf.default_opts()
    for k, v in kw.items():
        setattr(o, k, v)
    h = ctypes.c_void_p()
    rc = wf.lib.wf_plan(S, NC, H, D, W, ctypes.byref(o), ctypes.byref(h))
    return rc, h


def test_validation_codes():
    assert _plan(0, 48, 2, 32, -1, n_chunks=6)[0] == wf.WF_ERANGE
    assert _plan(9, 48, 2, 32, -1, n_chunks=6)[0] == wf.WF_ERANGE
    assert _plan(2, 48, 2, 30, -1, n_chunks=6)[0] == wf.WF_EINVAL       # D % 8
    assert _plan(2, 48, 2, 32, -2, n_chunks=6)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, grid_h=5, grid_w=4)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, dtype=7)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, anchor_mode=3)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, 1, n_chunks=6, store_extra_history=-1)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, store_extra_history=1)[0] == wf.WF_EINVAL   # full history
    assert _plan(2, 48, 2, 32, 3, n_chunks=6, store_extra_history=wf.WF_MAX_CTX)[0] == wf.WF_ERANGE
    # RoPE split: even parts >= 0 summing to head_dim, or all zero (default)
    for bad in ((15, 9, 8), (16, 8, 6), (-2, 18, 16), (34, 0, 0)):
        o = wf.default_opts()
        o.n_chunks = 6
        o.rope_split[0], o.rope_split[1], o.rope_split[2] = bad
        h = ctypes.c_void_p()
        assert wf.lib.wf_plan(2, 48, 2, 32, -1, ctypes.byref(o), ctypes.byref(h)) == wf.WF_EINVAL, bad
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, mask=2)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=6, schedule=2)[0] == wf.WF_EINVAL
    assert _plan(2, 48, 2, 32, -1, n_chunks=40)[0] == wf.WF_ERANGE      # context > 32 chunks
    assert wf.lib.wf_plan(2, 48, 2, 32, -1, None, None) == wf.WF_EINVAL
    rc, h = _plan(2, 48, 2, 32, -1, n_chunks=6, grid_h=4, grid_w=4)
    assert rc == wf.WF_OK
    try:
        n = ctypes.c_int()
        buf = (ctypes.c_int32 * 10)()
        assert wf.lib.wf_page_table(h, buf, 1, ctypes.byref(n)) == wf.WF_ENOROUND
        assert wf.lib.wf_qkv_rope_publish(h, 0, ctypes.c_void_p(256), None) == wf.WF_EUNBOUND
        assert wf.lib.wf_round_attention(h, 0, ctypes.c_void_p(256), 0, None) == wf.WF_EUNBOUND
        assert wf.lib.wf_bind(h, None, None, None) == wf.WF_EINVAL
        assert wf.lib.wf_bind(h, ctypes.c_void_p(256), ctypes.c_void_p(257),
                              ctypes.c_void_p(512)) == wf.WF_EINVAL
        info = wf.wf_round_info()
        for k in range(8):
            assert wf.lib.wf_round_step(h, ctypes.byref(info)) == wf.WF_OK
            assert info.k == k
        assert wf.lib.wf_round_step(h, ctypes.byref(info)) == wf.WF_EDONE
        assert info.k == 7
    finally:
        wf.lib.wf_plan_destroy(h)
    for c in (0, -1, -5, -10, -99):
        assert wf.lib.wf_strerror(c)


def test_buffer_sizes():
    rc, h = _plan(4, 4680, 12, 128, 3, n_chunks=133, layers=30, grid_h=30, grid_w=52)
    assert rc == 0
    s = wf.wf_buffer_sizes()
    assert wf.lib.wf_plan_buffer_sizes(h, ctypes.byref(s)) == 0
    # pages: anchor + (W+1) ring + S live + unrotated-anchor page (App. B.8)
    assert s.n_pages == 1 + 4 + 4 + 1 and s.ring_pages == 4
    tok = 4680 * 12 * 128 * 2
    assert s.qkv == 5 * 3 * tok and s.qbuf == 5 * tok and s.out == 5 * tok
    assert s.pool == 10 * 30 * 2 * tok
    wf.lib.wf_plan_destroy(h)


def _oracle_rows(cfg, k):
    rows = []
    for t in sch.round_tasks(cfg, k):
        for i, e in enumerate(t.context):
            rows.append((t.stage, t.chunk, t.stage, t.dest_page, i, e.kind, e.chunk, e.j, e.page, e.tpos))
    return rows


CFGS = [sch.Cfg(S, N, W, a, m) for S, N, W, a, m in itertools.product(
    [1, 2, 4, 5], [1, 3, 6, 12], [-1, 0, 1, 3], [True, False],
    [sch.ANCHOR_ADJACENT, sch.ANCHOR_ABSOLUTE])] + [sch.Cfg(4, 133, 3), sch.Cfg(5, 135, 3)]
# the comparison graphs: RF mask (wavefront rounds) and the sequential NF1C schedule
CFGS += [sch.Cfg(S, N, W, a, mask=sch.MASK_RF) for S, N, W, a in itertools.product(
    [1, 2, 4], [3, 12], [-1, 1, 3], [True, False])]
CFGS += [sch.Cfg(S, N, W, a, m, sequential=True) for S, N, W, a, m in itertools.product(
    [1, 2, 4], [1, 5], [-1, 0, 2], [True, False], [sch.ANCHOR_ADJACENT, sch.ANCHOR_ABSOLUTE])]
# the store's longer prefix (E extra history chunks for the store pass)
CFGS += [sch.Cfg(S, N, W, a, m, store_extra=E) for S, N, W, E, a, m in itertools.product(
    [1, 2, 4], [3, 12], [0, 1, 3], [1, 4], [True, False], [sch.ANCHOR_ADJACENT, sch.ANCHOR_ABSOLUTE])]
CFGS += [sch.Cfg(3, 12, 1, mask=sch.MASK_RF, store_extra=3), sch.Cfg(2, 5, 1, sequential=True, store_extra=2),
         sch.Cfg(4, 133, 3, store_extra=4)]


@pytest.mark.parametrize("cfg", CFGS, ids=str)
def test_page_table_bit_exact_vs_oracle(cfg):
    rc, h = _plan(cfg.S, 12, 1, 8, cfg.history, n_chunks=cfg.n_chunks, grid_h=2, grid_w=2,
                  use_anchor=int(cfg.use_anchor), anchor_mode=cfg.anchor_mode, mask=cfg.mask,
                  schedule=wf.WF_SCHED_SEQUENTIAL if cfg.sequential else wf.WF_SCHED_WAVEFRONT,
                  store_extra_history=cfg.store_extra)
    hist = cfg.history if cfg.history >= 0 else cfg.n_chunks - 1
    if 1 + hist + 1 + max(cfg.S, cfg.store_extra) > wf.WF_MAX_CTX:
        assert rc == wf.WF_ERANGE
        return
    assert rc == wf.WF_OK
    s = wf.wf_buffer_sizes()
    wf.lib.wf_plan_buffer_sizes(h, ctypes.byref(s))
    assert s.n_pages == sch.n_pages(cfg)
    try:
        info = wf.wf_round_info()
        cap = 512
        buf = (ctypes.c_int32 * (10 * cap))()
        n = ctypes.c_int()
        for k in range(sch.n_rounds(cfg)):
            assert wf.lib.wf_round_step(h, ctypes.byref(info)) == wf.WF_OK
            assert wf.lib.wf_page_table(h, buf, cap, ctypes.byref(n)) == wf.WF_OK
            got = [tuple(buf[10 * i:10 * i + 10]) for i in range(n.value)]
            assert got == _oracle_rows(cfg, k), f"round {k}"
            tasks = sch.round_tasks(cfg, k)
            assert info.n_tasks == len(tasks)
            u = sch.store_chunk(cfg, k)
            assert info.store_chunk == (u if u is not None else -1)
            fl = sum(4 * 12 * 12 * len(t.context) * 8 for t in tasks)
            assert info.attn_flops == fl
        assert wf.lib.wf_round_step(h, ctypes.byref(info)) == wf.WF_EDONE
    finally:
        wf.lib.wf_plan_destroy(h)


def test_dit_entry_points_validate_before_any_cuda_call():
    """The DiT and linear-layer entry points reject unbound plans and bad
    sizes on the host (no CUDA call is reached on these paths)."""
    rc, h = _plan(4, 4680, 12, 128, 3, n_chunks=64, grid_h=30, grid_w=52, layers=30)
    assert rc == wf.WF_OK
    try:
        n = ctypes.c_size_t()
        # model_dim must be heads * head_dim; ffn % 64; 4C % 64; freq even
        assert wf.lib.wf_dit_workspace_size(h, 1536, 8960, 16, 256, 0, ctypes.byref(n)) == wf.WF_OK
        rows = 5 * 4680
        lat = 16 * 3 * 60 * 104
        want = (rows * 1536 * 4 + rows * 1536 * 2 + rows * 8960 * 2 + rows * 64 * 2 + 2 * 5 * lat * 4
                + 30 * 5 * 6 * 1536 * 4 + 5 * 2 * 1536 * 4 + 5 * (256 + 9 * 1536) * 4)
        assert want <= n.value <= want + 16 * 256 + 30 * 128
        for bad in ((1535, 8960, 16, 256), (1536, 8961, 16, 256), (1536, 8960, 15, 256),
                    (1536, 8960, 16, 255)):
            assert wf.lib.wf_dit_workspace_size(h, *bad, 0, ctypes.byref(n)) == wf.WF_EINVAL
        assert wf.lib.wf_dit_workspace_size(h, 1536, 8960, 16, 256, 0, None) == wf.WF_EINVAL
        # e4m3 linear layers add the e4m3 activations and quantised weights
        n8 = ctypes.c_size_t()
        assert wf.lib.wf_dit_workspace_size(h, 1536, 8960, 16, 256, 1, ctypes.byref(n8)) == wf.WF_OK
        per_layer = 3 * 1536 * 1536 + 1536 * 1536 + 2 * 1536 * 8960
        assert n8.value - n.value >= rows * (1536 + 8960) + 30 * per_layer
        assert wf.lib.wf_dit_workspace_size(h, 1536, 8960, 16, 256, 2, ctypes.byref(n8)) == wf.WF_EINVAL
        m = wf.wf_dit_model()
        assert wf.lib.wf_dit_bind(h, ctypes.byref(m), ctypes.c_void_p(256), None) == wf.WF_EUNBOUND
        assert wf.lib.wf_dit_bind(h, None, ctypes.c_void_p(256), None) == wf.WF_EINVAL
        assert wf.lib.wf_dit_round(h, None, None, None, None, None) == wf.WF_EUNBOUND
        p = ctypes.c_void_p(256)
        assert wf.lib.wf_qkv_proj_rope_publish(h, 0, p, p, None, None, None, None, None) == wf.WF_EUNBOUND
        assert wf.lib.wf_linear(h, p, 128, 64, 0, 128, p, None, 64, 64, wf.WF_EPI_F32, p, 64,
                                None, 0, 1, None) == wf.WF_EUNBOUND
        assert wf.lib.wf_linear(None, p, 128, 64, 0, 128, p, None, 64, 64, wf.WF_EPI_F32, p, 64,
                                None, 0, 1, None) == wf.WF_EINVAL
    finally:
        wf.lib.wf_plan_destroy(h)


def test_group_entry_points_validate_on_the_host():
    """wf_group_create refuses unbound plans, bad counts and null
    arguments before any CUDA call; the launching calls refuse a null group."""
    plans = []
    for _ in range(2):
        rc, h = _plan(2, 48, 1, 32, 1, n_chunks=4, grid_h=4, grid_w=4)
        assert rc == wf.WF_OK
        plans.append(h)
    arr = (ctypes.c_void_p * 2)(plans[0].value, plans[1].value)
    g = ctypes.c_void_p()
    assert wf.lib.wf_group_create(arr, 2, ctypes.byref(g)) == wf.WF_EUNBOUND
    assert wf.lib.wf_group_create(arr, 0, ctypes.byref(g)) == wf.WF_ERANGE
    assert wf.lib.wf_group_create(arr, wf.WF_MAX_GROUP_PLANS + 1, ctypes.byref(g)) == wf.WF_ERANGE
    assert wf.lib.wf_group_create(None, 2, ctypes.byref(g)) == wf.WF_EINVAL
    assert wf.lib.wf_group_create(arr, 2, None) == wf.WF_EINVAL
    dup = (ctypes.c_void_p * 2)(plans[0].value, plans[0].value)
    assert wf.lib.wf_group_create(dup, 2, ctypes.byref(g)) == wf.WF_EINVAL
    assert g.value is None
    p = ctypes.c_void_p(256)
    assert wf.lib.wf_group_attention(None, 1, 0, p, wf.WF_ATTN_TC, None) == wf.WF_EINVAL
    assert wf.lib.wf_group_publish(None, 1, 0, p, None) == wf.WF_EINVAL
    assert wf.lib.wf_group_proj_publish(None, 1, 0, p, p, None, None, None, None, None) == wf.WF_EINVAL
    n = ctypes.c_size_t()
    assert wf.lib.wf_group_dit_workspace_size(None, 256, 512, 16, 256, 0, ctypes.byref(n)) == wf.WF_EINVAL
    assert wf.lib.wf_group_dit_bind(None, None, p, None) == wf.WF_EINVAL
    assert wf.lib.wf_group_dit_round(None, 1, p, p, None, None, None) == wf.WF_EINVAL
    wf.lib.wf_group_destroy(None)
    for h in plans:
        wf.lib.wf_plan_destroy(h)


def _round_plan(cfg, **kw):
    return _plan(cfg.S, 12, 1, 8, cfg.history, n_chunks=cfg.n_chunks, grid_h=2, grid_w=2,
                 use_anchor=int(cfg.use_anchor), anchor_mode=cfg.anchor_mode, mask=cfg.mask,
                 schedule=wf.WF_SCHED_SEQUENTIAL if cfg.sequential else wf.WF_SCHED_WAVEFRONT,
                 store_extra_history=cfg.store_extra, layers=3, **kw)


def _table(h):
    cap = 512
    buf = (ctypes.c_int32 * (10 * cap))()
    n = ctypes.c_int()
    assert wf.lib.wf_page_table(h, buf, cap, ctypes.byref(n)) == wf.WF_OK
    return [tuple(buf[10 * i:10 * i + 10]) for i in range(n.value)]


def _export(h):
    n = ctypes.c_size_t()
    assert wf.lib.wf_plan_state_size(h, ctypes.byref(n)) == wf.WF_OK
    buf = ctypes.create_string_buffer(n.value)
    w = ctypes.c_size_t()
    assert wf.lib.wf_plan_export_state(h, buf, n.value, ctypes.byref(w)) == wf.WF_OK
    assert w.value == n.value
    short = ctypes.create_string_buffer(n.value - 4)
    assert wf.lib.wf_plan_export_state(h, short, n.value - 4, ctypes.byref(w)) == wf.WF_ENOMEM
    return buf.raw


@pytest.mark.parametrize("cfg", [sch.Cfg(4, 14, 3), sch.Cfg(2, 7, -1), sch.Cfg(3, 9, 1, mask=sch.MASK_RF),
                                 sch.Cfg(2, 4, 1, sequential=True), sch.Cfg(3, 12, 1, store_extra=3)],
                         ids=str)
def test_state_export_import_resumes_the_request(cfg):
    """A request checkpointed at every round and resumed in a fresh plan
    follows the uninterrupted plan's schedule bit for bit to the end."""
    for cut in range(-1, sch.n_rounds(cfg)):
        rc, a = _round_plan(cfg)
        assert rc == wf.WF_OK
        for _ in range(cut + 1):
            assert wf.lib.wf_round_step(a, None) == wf.WF_OK
        state = _export(a)
        rc, b = _round_plan(cfg)
        assert wf.lib.wf_plan_import_state(b, state, len(state)) == wf.WF_OK
        if cut >= 0:
            assert _table(b) == _table(a)
        while True:
            ra, rb = wf.lib.wf_round_step(a, None), wf.lib.wf_round_step(b, None)
            assert ra == rb
            if ra == wf.WF_EDONE:
                break
            assert _table(a) == _table(b)
        wf.lib.wf_plan_destroy(a)
        wf.lib.wf_plan_destroy(b)


# word offsets of the checkpoint format: 22 shape words, then k,
# have_prev_store, prev_store_chunk, prev_store_page, anchor_stored, n_history
_SHAPE_WORDS = 22
_HEAD = _SHAPE_WORDS + 6


def _words(state):
    return list(memoryview(bytes(state)).cast("i"))


def _state(words):
    import array
    return array.array("i", words).tobytes()


def test_state_import_rejects_foreign_or_corrupt_state():
    cfg = sch.Cfg(4, 14, 3)
    rc, a = _round_plan(cfg)
    for _ in range(9):
        wf.lib.wf_round_step(a, None)
    state = bytearray(_export(a))
    rc, other = _plan(4, 12, 1, 8, 2, n_chunks=14, grid_h=2, grid_w=2, layers=3)   # W differs
    assert wf.lib.wf_plan_import_state(other, bytes(state), len(state)) == wf.WF_EINVAL
    rc, b = _round_plan(cfg)
    assert wf.lib.wf_plan_import_state(b, bytes(state[:-4]), len(state) - 4) == wf.WF_EINVAL
    w = _words(state)
    bad = list(w)
    bad[_HEAD] = 999                                                   # history chunk id
    assert wf.lib.wf_plan_import_state(b, _state(bad), len(state)) == wf.WF_EINVAL
    bad = bytearray(state)
    bad[0] ^= 1                                                       # magic
    assert wf.lib.wf_plan_import_state(b, bytes(bad), len(bad)) == wf.WF_EINVAL
    assert wf.lib.wf_plan_import_state(b, None, 0) == wf.WF_EINVAL
    assert wf.lib.wf_plan_import_state(b, bytes(state), len(state)) == wf.WF_OK
    assert wf.lib.wf_selftest_timeout(b, 1000, None) == wf.WF_EUNBOUND
    for h in (a, other, b):
        wf.lib.wf_plan_destroy(h)


def test_state_import_rejects_aliased_or_missing_pages():
    """Every ring page is in exactly one of history, the free list and the
    pending store page: a state that puts two chunks on one page (they would
    read each other's K/V) or loses a page is refused."""
    cfg = sch.Cfg(4, 14, 3)
    rc, a = _round_plan(cfg)
    for _ in range(9):        # k = 8: three history chunks, a pending store page
        wf.lib.wf_round_step(a, None)
    w = _words(_export(a))
    nh = w[_HEAD - 1]
    assert nh == 3 and w[_SHAPE_WORDS + 1] == 1
    hist_pages = [w[_HEAD + 2 * i + 1] for i in range(nh)]
    at_free = _HEAD + 2 * nh
    rc, b = _round_plan(cfg)
    # two history chunks on one page
    bad = list(w)
    bad[_HEAD + 3] = hist_pages[0]
    assert wf.lib.wf_plan_import_state(b, _state(bad), 4 * len(bad)) == wf.WF_EINVAL
    # the pending store page also in history
    bad = list(w)
    bad[_HEAD + 1] = w[_SHAPE_WORDS + 3]
    assert wf.lib.wf_plan_import_state(b, _state(bad), 4 * len(bad)) == wf.WF_EINVAL
    # a free page that is also in history (the ring has R = 4 pages, none free here)
    assert w[at_free] == 0
    bad = w[:at_free] + [1, hist_pages[1]] + w[at_free + 1:]
    assert wf.lib.wf_plan_import_state(b, _state(bad), 4 * len(bad)) == wf.WF_EINVAL
    # a page that belongs nowhere (the history list loses its oldest chunk)
    bad = list(w)
    bad[_HEAD - 1] = nh - 1
    del bad[_HEAD:_HEAD + 2]
    assert wf.lib.wf_plan_import_state(b, _state(bad), 4 * len(bad)) == wf.WF_EINVAL
    # history not oldest first
    bad = list(w)
    bad[_HEAD], bad[_HEAD + 2] = bad[_HEAD + 2], bad[_HEAD]
    assert wf.lib.wf_plan_import_state(b, _state(bad), 4 * len(bad)) == wf.WF_EINVAL
    assert wf.lib.wf_plan_import_state(b, _state(w), 4 * len(w)) == wf.WF_OK
    for h in (a, b):
        wf.lib.wf_plan_destroy(h)


@pytest.mark.parametrize("change", [dict(dtype=wf.WF_FP8), dict(rope_theta=500.0),
                                    dict(rope_split=(16, 8, 8)), dict(dtype=wf.WF_FP8, fp8_qk_scale=4.0)],
                         ids=["dtype", "theta", "split", "fp8_scale"])
def test_state_import_rejects_other_page_format(change):
    """A checkpoint resumes only into a plan whose pages hold the same bytes:
    same dtype, RoPE base and split, and the same e4m3 scales."""
    def plan(**kw):
        o = wf.default_opts()
        o.n_chunks, o.layers, o.grid_t, o.grid_h, o.grid_w = 9, 2, 3, 4, 4
        for k, v in kw.items():
            if k == "rope_split":
                o.rope_split[0], o.rope_split[1], o.rope_split[2] = v
            else:
                setattr(o, k, v)
        h = ctypes.c_void_p()
        assert wf.lib.wf_plan(2, 48, 1, 32, 2, ctypes.byref(o), ctypes.byref(h)) == wf.WF_OK
        return h
    base = dict(dtype=wf.WF_FP8) if "fp8_qk_scale" in change else {}
    a = plan(**base)
    for _ in range(5):
        assert wf.lib.wf_round_step(a, None) == wf.WF_OK
    st = _export(a)
    same, other = plan(**base), plan(**change)
    assert wf.lib.wf_plan_import_state(same, st, len(st)) == wf.WF_OK
    assert wf.lib.wf_plan_import_state(other, st, len(st)) == wf.WF_EINVAL
    for h in (a, same, other):
        wf.lib.wf_plan_destroy(h)


def test_rope_split_sizes_the_tables():
    """A custom split changes exactly the rotary tables in scratch: 8 bytes
    per (position, pair) of each part (t over all chunks' frames, h, w)."""
    def scratch(split):
        o = wf.default_opts()
        o.n_chunks, o.grid_t, o.grid_h, o.grid_w = 5, 3, 4, 4
        if split:
            o.rope_split[0], o.rope_split[1], o.rope_split[2] = split
        h = ctypes.c_void_p()
        assert wf.lib.wf_plan(2, 48, 1, 32, 1, ctypes.byref(o), ctypes.byref(h)) == wf.WF_OK
        s = wf.wf_buffer_sizes()
        assert wf.lib.wf_plan_buffer_sizes(h, ctypes.byref(s)) == wf.WF_OK
        wf.lib.wf_plan_destroy(h)
        return s.scratch
    t_max, gh, gw = 3 * 5, 4, 4
    pairs = lambda dt, dh, dw: t_max * dt // 2 + gh * dh // 2 + gw * dw // 2
    base = scratch(None)
    assert scratch((12, 10, 10)) == base                  # the default split for D = 32
    for split in ((32, 0, 0), (16, 8, 8), (0, 16, 16)):
        assert scratch(split) - base == 8 * (pairs(*split) - pairs(12, 10, 10)), split
