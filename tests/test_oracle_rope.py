"""Pins of the fp64 3D RoPE: rotation invariants and closed forms.

The paper fixes only that RoPE is applied after the QKV projection and that
the anchor's key is re-rotated when the window shifts ("Wave Forcing"
Sec. 4.2, App. B.3); the convention (split, base, pairs) is a reading, so
these tests pin the mathematics of the rotation, not the convention.
"""

import numpy as np
import pytest

from oracle import rope


def test_sections():
    assert rope.sections(128) == (44, 42, 42)
    assert rope.sections(32) == (12, 10, 10)
    assert sum(rope.sections(64)) == 64


def test_identity_at_origin_and_first_pair_closed_form():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((1, 2, 128))
    z = rope.rotate(x, rope.pair_angles(128, 1e4, [0], [0], [0]))
    assert np.array_equal(z, x)
    # pair 0 of the temporal part has frequency theta^0 = 1: angle = t
    e0 = np.zeros((1, 128))
    e0[0, 0] = 1.0
    for t in (1, 5, 17):
        y = rope.rotate(e0, rope.pair_angles(128, 1e4, [t], [0], [0]))
        assert y[0, 0] == pytest.approx(np.cos(t), abs=1e-15)
        assert y[0, 1] == pytest.approx(np.sin(t), abs=1e-15)
        assert np.count_nonzero(y[0, 2:]) == 0
    # first pair of the height part (channels 44, 45) rotates by h
    e = np.zeros((1, 128))
    e[0, 45] = 1.0
    y = rope.rotate(e, rope.pair_angles(128, 1e4, [3], [2], [9]))
    assert y[0, 44] == pytest.approx(-np.sin(2), abs=1e-15)
    assert y[0, 45] == pytest.approx(np.cos(2), abs=1e-15)
    # last pair of the width part: angle = w * theta^(-(d-2)/d), d = 42
    e = np.zeros((1, 128))
    e[0, 126] = 1.0
    y = rope.rotate(e, rope.pair_angles(128, 1e4, [0], [0], [7]))
    a = 7 * 1e4 ** (-40.0 / 42.0)
    assert y[0, 126] == pytest.approx(np.cos(a), abs=1e-15)
    assert y[0, 127] == pytest.approx(np.sin(a), abs=1e-15)


def test_norm_preserved_per_pair():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 3, 128))
    t, h, w = rng.integers(0, 400, 50), rng.integers(0, 30, 50), rng.integers(0, 52, 50)
    y = rope.rotate(x, rope.pair_angles(128, 1e4, t, h, w))
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(nx, ny, rtol=1e-13, atol=1e-13)


def test_relative_position():
    # q.k depends only on the position difference along each axis
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))

    def dot(pq, pk):
        a = rope.rotate(q, rope.pair_angles(128, 1e4, *[[v] for v in pq]))
        b = rope.rotate(k, rope.pair_angles(128, 1e4, *[[v] for v in pk]))
        return float((a * b).sum())

    base = dot((10, 4, 7), (3, 1, 20))
    assert dot((110, 4, 7), (103, 1, 20)) == pytest.approx(base, rel=1e-11, abs=1e-11)
    assert dot((10, 14, 27), (3, 11, 40)) == pytest.approx(base, rel=1e-11, abs=1e-11)
    assert dot((10, 4, 7), (4, 1, 20)) != pytest.approx(base, rel=1e-6)


def test_rerotation_composes():
    # anchor re-rotation (App. B.3): rotating the unrotated key at the new
    # position equals rotating the old rotated key by the position difference
    rng = np.random.default_rng(3)
    k = rng.standard_normal((48, 2, 32))
    grid = (3, 4, 4)
    at0 = rope.rope_chunk(k, 0, grid, 1e4)
    at5 = rope.rope_chunk(k, 5, grid, 1e4)
    t, h, w = rope.chunk_positions(5, *grid)
    t0, _, _ = rope.chunk_positions(0, *grid)
    delta = rope.pair_angles(32, 1e4, t - t0, np.zeros_like(h), np.zeros_like(w))
    assert np.allclose(rope.rotate(at0, delta), at5, atol=1e-12)


def test_chunk_positions_layout():
    t, h, w = rope.chunk_positions(2, 3, 30, 52)
    assert len(t) == 4680
    assert (t[0], h[0], w[0]) == (6, 0, 0)
    assert (t[1559], h[1559], w[1559]) == (6, 29, 51)
    assert (t[1560], h[1560], w[1560]) == (7, 0, 0)
    assert (t[53], h[53], w[53]) == (6, 1, 1)


# ---- a custom (d_t, d_h, d_w) split (plan option) ----------------------------------

def test_custom_split_equal_to_default_changes_nothing():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((60, 2, 128))
    assert np.array_equal(rope.rope_chunk(x, 4, (3, 4, 5), 1e4),
                          rope.rope_chunk(x, 4, (3, 4, 5), 1e4, split=(44, 42, 42)))


def test_temporal_only_split_is_one_dimensional_rope():
    """(D, 0, 0): every pair rotates by t * theta^(-2m/D), the textbook 1-D
    rotary embedding of the frame index; tokens of one frame rotate alike."""
    D, theta = 32, 1e4
    rng = np.random.default_rng(4)
    x = rng.standard_normal((24, 1, D))
    y = rope.rope_chunk(x, 2, (3, 2, 4), theta, split=(D, 0, 0))
    t = 3 * 2 + np.arange(24) // 8
    for n in range(24):
        for m in range(D // 2):
            a = t[n] * theta ** (-2.0 * m / D)
            c, s = np.cos(a), np.sin(a)
            x0, x1 = x[n, 0, 2 * m], x[n, 0, 2 * m + 1]
            assert np.isclose(y[n, 0, 2 * m], x0 * c - x1 * s, rtol=0, atol=1e-12)
            assert np.isclose(y[n, 0, 2 * m + 1], x0 * s + x1 * c, rtol=0, atol=1e-12)


def test_custom_split_parts_follow_their_axes():
    """With split (d_t, d_h, d_w) the pairs of each part depend only on that
    axis' coordinate: moving a token along w leaves the t and h parts alone."""
    D, split = 64, (16, 32, 16)
    ang_a = rope.pair_angles(D, 1e4, [5], [2], [1], split)
    ang_b = rope.pair_angles(D, 1e4, [5], [2], [7], split)
    nt, nh = split[0] // 2, split[1] // 2
    assert np.array_equal(ang_a[:, :nt + nh], ang_b[:, :nt + nh])
    assert not np.array_equal(ang_a[:, nt + nh:], ang_b[:, nt + nh:])
    x = np.random.default_rng(5).standard_normal((1, 1, D))
    for sp in (split, (64, 0, 0), (0, 0, 64)):
        y = rope.rotate(x, rope.pair_angles(D, 1e4, [3], [1], [2], sp))
        assert np.allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]))


@pytest.mark.parametrize("bad", [(15, 9, 8), (16, 8, 6), (-2, 18, 16)])
def test_bad_split_is_rejected(bad):
    with pytest.raises(ValueError):
        rope.sections(32, bad)
