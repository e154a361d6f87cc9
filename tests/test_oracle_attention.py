"""Pins of the oracle's attention: textbook/library reductions, closed forms,
invariants and Proposition 1 ("Wave Forcing" Sec. 3.1 Eq. 4-5, App. B.6)."""

import math

import numpy as np
import pytest
import torch

from oracle import schedule as sch
from oracle.attention import masked_attention, masked_softmax
from oracle.round import Geom, round_attention, round_attention_replay, round_universe
import wf_synth


def test_masked_attention_matches_library_sdpa():
    rng = np.random.default_rng(0)
    H, nq, nk, D = 3, 7, 11, 16
    q, k, v = (rng.standard_normal((H, n, D)) for n in (nq, nk, nk))
    mask = rng.random((nq, nk)) < 0.6
    mask[:, 0] = True
    ours = masked_attention(q, k, v, mask)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask)).numpy()
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-13)


def test_masked_attention_brute_force_loops():
    rng = np.random.default_rng(1)
    nq, nk, D = 4, 5, 3
    q, k, v = (rng.standard_normal((1, n, D)) for n in (nq, nk, nk))
    mask = np.array([[1, 0, 1, 1, 0], [1, 1, 1, 1, 1], [0, 0, 0, 0, 1], [1, 1, 0, 0, 0]], bool)
    ours = masked_attention(q, k, v, mask)[0]
    for i in range(nq):
        w = [math.exp(sum(q[0, i, d] * k[0, j, d] for d in range(D)) / math.sqrt(D))
             if mask[i, j] else 0.0 for j in range(nk)]
        z = sum(w)
        for d in range(D):
            assert ours[i, d] == pytest.approx(sum(w[j] * v[0, j, d] for j in range(nk)) / z,
                                               rel=1e-12, abs=1e-14)


def test_softmax_rows_sum_to_one_and_masked_are_zero():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((5, 9)) * 30
    m = rng.random((5, 9)) < 0.5
    m[:, 3] = True
    p = masked_softmax(s, m)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)
    assert np.all(p[~m] == 0.0)


GEOM = Geom(grid_t=3, grid_h=2, grid_w=2, heads=2, head_dim=8)


def _raw_random(seed):
    def raw(chunk, stage, layer):
        return wf_synth.qkv_raw(seed, chunk, stage, layer, GEOM.chunk_tokens,
                                GEOM.heads, GEOM.head_dim).double().numpy()
    return raw


CFGS = [sch.Cfg(2, 6, -1), sch.Cfg(4, 10, 3), sch.Cfg(3, 7, 1, anchor_mode=sch.ANCHOR_ABSOLUTE),
        sch.Cfg(3, 5, 2, use_anchor=False),
        # the store keeps E more history chunks than the denoising tasks
        sch.Cfg(4, 11, 2, store_extra=4), sch.Cfg(3, 8, 1, store_extra=1),
        sch.Cfg(2, 7, 0, store_extra=2, use_anchor=False), sch.Cfg(2, 5, 1, sequential=True, store_extra=2)]


@pytest.mark.parametrize("cfg", CFGS, ids=str)
def test_batched_mask_equals_sequential_replay(cfg):
    """Proposition 1: dependency-respecting sequential execution over the
    ordered contexts equals the batched (mask) execution."""
    raw = _raw_random(11)
    for k in range(sch.n_rounds(cfg)):
        a = round_attention(cfg, GEOM, k, 0, raw)
        b = round_attention_replay(cfg, GEOM, k, 0, raw)
        assert len(a) == len(b) == len(sch.round_tasks(cfg, k))
        for x, y in zip(a, b):
            assert np.allclose(x, y, rtol=1e-12, atol=1e-13)


def _fingerprint_raw(cfg):
    """Q = 0 (uniform softmax over visible keys), V = one-hot of the producing
    (chunk, stage), so O[:, :, c] = share of visible tokens from chunk c."""
    D = GEOM.head_dim * 4

    def raw(chunk, stage, layer):
        x = np.zeros((GEOM.chunk_tokens, 3, GEOM.heads, D))
        rng = np.random.default_rng(chunk * 31 + stage)
        x[:, 1] = rng.standard_normal(x[:, 1].shape)
        x[:, 2, :, chunk] = 1.0
        x[:, 2, :, 16 + stage] = 1.0
        return x
    return raw, Geom(GEOM.grid_t, GEOM.grid_h, GEOM.grid_w, GEOM.heads, D)


@pytest.mark.parametrize("cfg", CFGS, ids=str)
def test_visibility_fingerprint_closed_form(cfg):
    raw, geom = _fingerprint_raw(cfg)
    for k in range(sch.n_rounds(cfg)):
        outs = round_attention(cfg, geom, k, 0, raw)
        for t, o in zip(sch.round_tasks(cfg, k), outs):
            want = np.zeros(geom.head_dim)
            n = len(t.context)
            for e in t.context:
                stage = e.j if e.kind == sch.KIND_LIVE else cfg.S
                want[e.chunk] += 1.0 / n
                want[16 + stage] += 1.0 / n
            assert np.allclose(o, want[None, None, :], atol=1e-14), (k, t.chunk, t.stage)


def test_zero_query_is_mean_of_visible_values():
    cfg = sch.Cfg(4, 10, 3)
    rnd = _raw_random(5)

    def raw(chunk, stage, layer):
        x = rnd(chunk, stage, layer).copy()
        x[:, 0] = 0.0
        return x
    k = 9
    outs = round_attention(cfg, GEOM, k, 0, raw)
    for t, o in zip(sch.round_tasks(cfg, k), outs):
        vs = [raw(e.chunk, e.j if e.kind == sch.KIND_LIVE else cfg.S, 0)[:, 2] for e in t.context]
        mean = np.concatenate(vs, axis=0).mean(axis=0)
        assert np.allclose(o, mean[None], atol=1e-13)


def test_sampled_rows_match_full():
    cfg = sch.Cfg(4, 10, 3)
    raw = _raw_random(3)
    uni = round_universe(cfg, GEOM, 9, 0, raw)
    full = round_attention(cfg, GEOM, 9, 0, raw, universe=uni)
    rows = [0, 5, 11]
    part = round_attention(cfg, GEOM, 9, 0, raw, rows=rows, universe=uni)
    for a, b in zip(full, part):
        assert np.array_equal(a[rows], b)


def test_planted_mask_mistake_is_caught():
    """Dropping self-visibility (j > s instead of Eq. 4's j >= s) or letting the
    store see live chunks must break the closed-form fingerprint."""
    cfg = sch.Cfg(2, 6, -1)
    raw, geom = _fingerprint_raw(cfg)
    k = 3
    K, V, lab, _, _ = round_universe(cfg, geom, k, 0, raw)
    q0 = np.zeros((geom.heads, 1, geom.head_dim))
    for t in sch.round_tasks(cfg, k):
        want = np.zeros(geom.head_dim)
        for e in t.context:
            want[e.chunk] += 1.0 / len(t.context)
            want[16 + (e.j if e.kind == sch.KIND_LIVE else cfg.S)] += 1.0 / len(t.context)
        good = masked_attention(q0, K, V, (lab >= t.stage)[None, :])
        assert np.allclose(good[:, 0], want[None], atol=1e-14)
        wrong_masks = [lab > t.stage, lab >= 0]
        if t.stage > 0:
            wrong_masks.append(lab >= t.stage - 1)
        for m in wrong_masks:
            if m.any() and not np.array_equal(m, lab >= t.stage):
                bad = masked_attention(q0, K, V, m[None, :])
                assert not np.allclose(bad[:, 0], want[None], atol=1e-6)


def test_bf16_rounding_of_attention_inputs():
    """round_to('bf16') is IEEE round-to-nearest-even onto 8 significant bits."""
    from oracle.round import round_to
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7, -3.0 - 2 ** -7, 2 ** -130 * 3])
    want = np.array([1.0, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -3.0, 2 ** -130 * 3])
    assert np.array_equal(round_to(x, "bf16"), want)
    assert round_to(x, None) is x
    y = np.random.default_rng(0).standard_normal(1000)
    r = round_to(y, "bf16")
    assert np.all(np.abs(r - y) <= 2.0 ** -8 * np.abs(y))


# ---- 8-bit (e4m3) storage -------------------------------------------------------

def test_e4m3_rounding_matches_the_format_definition():
    """OCP FP8 e4m3 (4 exponent bits, bias 7, 3 mantissa bits, no infinity,
    max 448): spacing 1/8 on [1, 2), round to nearest even, subnormals in
    steps of 2^-9, saturation at 448 (satfinite)."""
    from oracle.round import e4m3
    cases = {1.0625: 1.0,            # halfway 1 .. 1.125 -> even (1.000b)
             1.1875: 1.25,           # halfway 1.125 .. 1.25 -> even (1.010b)
             1.1: 1.125, -3.3: -3.25, 448.0: 448.0, 500.0: 448.0, -1e4: -448.0,
             2.0 ** -6: 2.0 ** -6,   # smallest normal
             2.0 ** -9: 2.0 ** -9,   # smallest subnormal
             2.0 ** -10: 0.0,        # halfway 0 .. 2^-9 -> even (0)
             3 * 2.0 ** -10: 2 * 2.0 ** -9, 0.0: 0.0}
    for x, want in cases.items():
        assert e4m3(np.array([x]))[0] == want, x
    # the scale multiplies before and divides after the rounding
    assert e4m3(np.array([0.3]), 8.0)[0] == 2.5 / 8.0


def test_fp8_fingerprint_is_exact():
    """With Q = 0 and V one-hot in {0, 1} (exact in e4m3) the 8-bit round
    still yields O = 1/|context| per visible entry (up to fp64 rounding): the mask and
    page bookkeeping are unaffected by the storage precision."""
    from oracle.round import Fp8, round_attention
    cfg = sch.Cfg(3, 7, 2)
    geom = Geom(1, 2, 3, 1, 16)
    n = geom.chunk_tokens

    def raw(c, s, l):
        x = np.zeros((n, 3, 1, 16))
        x[:, 1] = np.random.default_rng(100 * c + s).normal(size=(n, 1, 16))
        x[:, 2, :, c] = 1.0
        return x

    k = 6
    outs = round_attention(cfg, geom, k, 0, raw, qk_dtype=Fp8(4.0, 1.0))
    for t, o in zip(sch.round_tasks(cfg, k), outs):
        want = np.zeros(16)
        for e in t.context:
            want[e.chunk] += 1.0 / len(t.context)
        assert np.allclose(o[:, 0, :], np.broadcast_to(want, (n, 16)), rtol=0, atol=1e-14)
