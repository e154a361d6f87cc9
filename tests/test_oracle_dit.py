"""Pins of the fp64 DiT oracle (oracle/dit.py) against facts fixed outside it:
closed forms, library routines written differently (torch conv3d, layer_norm,
gelu, scaled_dot_product_attention), invariants, and the sequential replay of
App. B.6 Proposition 1."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import wf_synth
from oracle import dit
from oracle import schedule as sch
from oracle.rope import rope_chunk

SMALL = dit.Dims(dim=64, heads=2, head_dim=32, ffn=96, layers=2, channels=4, freq=32)
GRID = (3, 2, 3)
STEPS4 = [1000.0, 750.0, 500.0, 250.0]


def model(cfg, dims=SMALL, grid=GRID, seed=3, bf16_points=False, steps=None, params=None):
    params = params or wf_synth.dit_params(seed, dims.dim, dims.ffn, dims.layers, dims.channels,
                                           dims.freq, std=0.2)
    return dit.Model(cfg, grid, dims, dit.weights_from(params), steps or STEPS4[:cfg.S],
                     bf16_points=bf16_points)


def lat(seed, c, s, dims=SMALL, grid=GRID):
    return wf_synth.latent(seed, c, s, dims.channels, grid[0], 2 * grid[1], 2 * grid[2]).double().numpy()


# ---- elementwise pieces -------------------------------------------------------

def test_layer_norm_matches_torch_and_is_standardised():
    x = np.random.default_rng(0).normal(size=(7, 48)) * 3 + 1
    y = dit.layer_norm(x)
    ref = F.layer_norm(torch.from_numpy(x), (48,), eps=1e-6).numpy()
    assert np.allclose(y, ref, atol=1e-12)
    assert np.allclose(y.mean(-1), 0, atol=1e-12)
    assert np.allclose((y ** 2).mean(-1), 1, atol=1e-5)


def test_rms_norm_matches_torch_and_closed_forms():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(6, 48)) * 3 + 0.5
    g = 1 + 0.3 * rng.normal(size=48)
    y = dit.rms_norm(x, g)
    ref = F.rms_norm(torch.from_numpy(x), (48,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    assert np.allclose(y, ref, atol=1e-12)
    # unit gain: mean square m / (m + eps) per row
    y1 = dit.rms_norm(x, np.ones(48))
    m = (x * x).mean(-1)
    assert np.allclose((y1 * y1).mean(-1), m / (m + 1e-6), atol=1e-13)
    # a constant row c maps to c / sqrt(c^2 + eps) times the gain
    for c in (-2.5, 1e-3, 7.0):
        row = dit.rms_norm(np.full(48, c), g)
        assert np.allclose(row, c / math.sqrt(c * c + 1e-6) * g, atol=1e-14)
    assert np.array_equal(dit.rms_norm(np.zeros(48), g), np.zeros(48))


def test_qk_norm_spans_the_full_width():
    """The q/k RMSNorm of the block normalises all heads of a token together:
    heads whose projections differ in size by 8x still differ by 8x after
    the norm and RoPE (a per-head norm would equalise them)."""
    cfg = sch.Cfg(S=1, n_chunks=1, history=-1)
    params = wf_synth.dit_params(5, SMALL.dim, SMALL.ffn, SMALL.layers, SMALL.channels,
                                 SMALL.freq, std=0.2)
    hd = SMALL.head_dim
    for name in ("nq", "nk"):
        params[name][0] = torch.ones(SMALL.dim, dtype=torch.bfloat16)
    w = params["qkv_w"][0].clone()
    w[hd:2 * hd] = w[:hd] * 8                               # q head 1 = 8 x q head 0 (exact in bf16)
    w[SMALL.dim + hd:SMALL.dim + 2 * hd] = w[SMALL.dim:SMALL.dim + hd] * 8
    params["qkv_w"][0] = w
    params["qkv_b"][0] = torch.zeros(3 * SMALL.dim, dtype=torch.bfloat16)
    m = model(cfg, params=params, steps=[1000.0])
    q, k, _, kraw = m.qkv(m.embed(lat(9, 0, -1)), 0, 0, 0)
    for t in (q, k, kraw):
        r = np.linalg.norm(t[:, 1], axis=-1) / np.linalg.norm(t[:, 0], axis=-1)
        assert np.allclose(r, 8.0, rtol=1e-9)
        assert np.allclose((t ** 2).mean(axis=(1, 2)), 1.0, atol=1e-5)   # unit RMS over the width


def test_gelu_tanh_odd_identity_and_torch():
    x = np.linspace(-6, 6, 241)
    g = dit.gelu_tanh(x)
    # 0.5 x (1 + tanh u) - 0.5 (-x)(1 + tanh(-u)) = x exactly for the tanh form
    assert np.allclose(g - dit.gelu_tanh(-x), x, atol=1e-13)
    assert dit.gelu_tanh(np.array([0.0]))[0] == 0.0
    ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(g, ref, atol=1e-12)


def test_silu_closed_forms():
    assert dit.silu(np.array([0.0]))[0] == 0.0
    assert np.isclose(dit.silu(np.array([1.0]))[0], 1.0 / (1.0 + math.exp(-1.0)))
    x = np.linspace(-5, 5, 11)
    assert np.allclose(dit.silu(x), F.silu(torch.from_numpy(x)).numpy(), atol=1e-14)


def test_sinusoid_closed_forms():
    e0 = dit.sinusoid(0.0, 256)
    assert np.array_equal(e0, np.concatenate([np.ones(128), np.zeros(128)]))
    t = 937.5
    e = dit.sinusoid(t, 256)
    assert np.isclose(e[0], math.cos(t)) and np.isclose(e[128], math.sin(t))
    assert np.allclose(e[:128] ** 2 + e[128:] ** 2, 1.0)
    # the last frequency is 10000^(-127/128)
    assert np.isclose(e[127], math.cos(t * 10000.0 ** (-127 / 128)))


def test_warp_sigma_shift5_values():
    # sigma' = 5 sigma / (1 + 4 sigma) (App. A, shift factor 5)
    assert dit.warp_sigma(1000) == 1.0
    assert dit.warp_sigma(0) == 0.0
    assert math.isclose(dit.warp_sigma(500), 5 / 6)
    assert math.isclose(dit.warp_sigma(250), 0.625)
    assert math.isclose(dit.warp_sigma(750), 3.75 / 4)
    # monotone: the warped schedule keeps nu_0 > ... > nu_{S-1} ordered
    s = [dit.warp_sigma(v) for v in [1000, 800, 600, 400, 200]]
    assert all(a > b for a, b in zip(s, s[1:]))


def test_psi_endpoints():
    x = np.random.default_rng(1).normal(size=(4, 5))
    e = np.random.default_rng(2).normal(size=(4, 5))
    assert np.array_equal(dit.psi(x, e, 0.0), x)            # Psi_0 = identity (Eq. 1)
    assert np.allclose(dit.psi(x, e, 1000.0), e)            # pure noise at nu = 1000
    s = dit.warp_sigma(500)
    assert np.allclose(dit.psi(x, e, 500.0), (1 - s) * x + s * e)


# ---- patches -----------------------------------------------------------------------

def test_patch_embedding_equals_strided_conv3d():
    rng = np.random.default_rng(4)
    C, Fr, gh, gw, dim = 4, 3, 2, 3, 8
    z = rng.normal(size=(C, Fr, 2 * gh, 2 * gw))
    w = rng.normal(size=(dim, C, 1, 2, 2))
    rows = dit.patchify(z) @ w.reshape(dim, -1).T               # [F gh gw, dim]
    conv = F.conv3d(torch.from_numpy(z)[None], torch.from_numpy(w), stride=(1, 2, 2))[0]
    ref = conv.numpy().reshape(dim, -1).T                        # tokens f, h, w
    assert np.allclose(rows, ref, atol=1e-12)


def test_unpatchify_places_each_output():
    C, Fr, gh, gw = 3, 2, 2, 3
    n = Fr * gh * gw
    y = np.arange(n * 4 * C, dtype=np.float64).reshape(n, 4 * C)
    z = dit.unpatchify(y, C, Fr, gh, gw)
    for tok in range(n):
        f, h, w = tok // (gh * gw), (tok // gw) % gh, tok % gw
        for q in range(2):
            for r in range(2):
                for c in range(C):
                    assert z[c, f, 2 * h + q, 2 * w + r] == y[tok, (2 * q + r) * C + c]


# ---- one block against library routines ----------------------------------------------

def torch_dense_forward(params, dims, grid, z, t_model, theta=10000.0):
    """The same Wan-style forward of one chunk with full (bidirectional)
    attention, written with torch fp64 library calls."""
    D = torch.float64
    P = {k: ([x.to(D) for x in v] if isinstance(v, list) else v.to(D)) for k, v in params.items()}
    zt = torch.from_numpy(z)
    C, Fr, gh, gw = dims.channels, grid[0], grid[1], grid[2]
    w5 = P["patch_w"].reshape(dims.dim, C, 1, 2, 2)
    x = F.conv3d(zt[None], w5, bias=P["patch_b"], stride=(1, 2, 2))[0]
    x = x.reshape(dims.dim, -1).T                                  # [N, dim]
    half = dims.freq // 2
    freqs = torch.pow(torch.tensor(10000.0, dtype=D), -torch.arange(half, dtype=D) / half)
    sin = torch.cat([torch.cos(t_model * freqs), torch.sin(t_model * freqs)])
    e = F.linear(F.silu(F.linear(sin, P["t1_w"], P["t1_b"])), P["t2_w"], P["t2_b"])
    e0 = F.linear(F.silu(e), P["tp_w"], P["tp_b"]).reshape(6, dims.dim)
    n = x.shape[0]
    for l in range(dims.layers):
        m = P["mod"][l] + e0
        xa = F.layer_norm(x, (dims.dim,), eps=1e-6) * (1 + m[1]) + m[0]
        qkv = F.linear(xa, P["qkv_w"][l], P["qkv_b"][l])
        q, k, v = qkv.split(dims.dim, dim=1)
        q = F.rms_norm(q, (dims.dim,), weight=P["nq"][l], eps=1e-6)
        k = F.rms_norm(k, (dims.dim,), weight=P["nk"][l], eps=1e-6)
        q = torch.from_numpy(rope_chunk(q.reshape(n, dims.heads, -1).numpy(), 0, grid, theta))
        k = torch.from_numpy(rope_chunk(k.reshape(n, dims.heads, -1).numpy(), 0, grid, theta))
        v = v.reshape(n, dims.heads, -1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1))
        o = o.transpose(0, 1).reshape(n, dims.dim)
        x = x + m[2] * F.linear(o, P["o_w"][l], P["o_b"][l])
        xf = F.layer_norm(x, (dims.dim,), eps=1e-6) * (1 + m[4]) + m[3]
        x = x + m[5] * F.linear(F.gelu(F.linear(xf, P["f1_w"][l], P["f1_b"][l]), approximate="tanh"),
                                P["f2_w"][l], P["f2_b"][l])
    hm = P["head_mod"] + e[None]
    y = F.linear(F.layer_norm(x, (dims.dim,), eps=1e-6) * (1 + hm[1]) + hm[0], P["head_w"], P["head_b"])
    # (row off, col off, channel) features back onto the latent grid
    y = y.reshape(Fr, gh, gw, 2, 2, C).permute(5, 0, 1, 3, 2, 4).reshape(C, Fr, 2 * gh, 2 * gw)
    return y.numpy()


def test_single_chunk_single_step_equals_dense_library_forward():
    """S = 1, one chunk: round 0 runs stage 0 of chunk 0 alone, attending to
    itself only -- a plain bidirectional transformer forward."""
    cfg = sch.Cfg(S=1, n_chunks=1, history=-1)
    params = wf_synth.dit_params(5, SMALL.dim, SMALL.ffn, SMALL.layers, SMALL.channels,
                                 SMALL.freq, std=0.2)
    m = model(cfg, params=params, steps=[1000.0])
    z = lat(9, 0, -1)
    x0s, emitted = m.round(0, z, [None])
    ref = torch_dense_forward(params, SMALL, GRID, z, 1000.0 * dit.warp_sigma(1000.0))
    assert np.allclose(x0s[0], ref, atol=1e-10), np.abs(x0s[0] - ref).max()
    assert emitted is not None and np.array_equal(emitted, x0s[0])  # Psi_0 = identity


def test_zero_gates_leave_the_residual_stream_alone():
    cfg = sch.Cfg(S=1, n_chunks=1, history=-1)
    params = wf_synth.dit_params(6, SMALL.dim, SMALL.ffn, SMALL.layers, SMALL.channels,
                                 SMALL.freq, std=0.2)
    for l in range(SMALL.layers):
        params["mod"][l].zero_()
    params["tp_w"].zero_()
    params["tp_b"].zero_()                      # e0 = 0 -> every gate is 0
    m = model(cfg, params=params, steps=[1000.0])
    z = lat(9, 0, -1)
    x = m.embed(z)
    for l in range(SMALL.layers):
        q, k, v, _ = m.qkv(x, 0, l, 0)
        o = np.random.default_rng(l).normal(size=(x.shape[0], SMALL.heads, SMALL.head_dim))
        assert np.array_equal(m.finish_layer(x, o, 0, l), x)


# ---- the round ---------------------------------------------------------------------

@pytest.mark.parametrize("S,n,W,E", [(2, 5, -1, 0), (2, 6, 1, 0), (3, 7, 2, 0), (2, 7, 1, 2)])
@pytest.mark.parametrize("bf16_points", [False, True])
def test_layer_major_masked_round_equals_sequential_replay(S, n, W, E, bf16_points):
    """App. B.6 Proposition 1: the batched, masked layer-major round equals
    task-at-a-time execution over the ordered contexts, round after round
    (E: history kept by the store only, label S + 2 in the mask)."""
    cfg = sch.Cfg(S=S, n_chunks=n, history=W, store_extra=E)
    a = model(cfg, bf16_points=bf16_points)
    b = model(cfg, bf16_points=bf16_points)
    for k in range(sch.n_rounds(cfg)):
        z = lat(11, k, -1)
        eps = [lat(11, k - s, s) for s in range(S)]
        xa, ea = a.round(k, z, eps)
        xb, eb = b.round_replay(k, z, eps)
        for u, v in zip(xa, xb):
            assert np.allclose(u, v, atol=1e-10), (k, np.abs(u - v).max())
        assert (ea is None) == (eb is None)
        if ea is not None:
            assert np.allclose(ea, eb, atol=1e-10)


def test_one_chunk_emitted_per_round_after_fill_in_order():
    S, n = 3, 6
    cfg = sch.Cfg(S=S, n_chunks=n, history=2)
    m = model(cfg)
    emitted = []
    for k in range(sch.n_rounds(cfg)):
        _, e = m.round(k, lat(2, k, -1), [lat(2, k - s, s) for s in range(S)])
        emitted.append(e is not None)
    # chunk i leaves stage S-1 in round i + S - 1 (Eq. 3)
    assert emitted == [S - 1 <= k < n + S - 1 for k in range(n + S)]


def test_history_is_read_not_recomputed():
    """A cached chunk's K/V are those its store pass produced: perturbing the
    current round's live inputs of other chunks cannot change the store task's
    output (it sees only anchor, history and itself, App. B.3)."""
    S, n = 2, 6
    cfg = sch.Cfg(S=S, n_chunks=n, history=1)
    a, b = model(cfg), model(cfg)
    k_end = 5
    for k in range(k_end + 1):
        z = lat(4, k, -1)
        eps = [lat(4, k - s, s) for s in range(S)]
        xa, _ = a.round(k, z, eps)
        zb = z + (10.0 if k == k_end else 0.0)          # only chunk k's fresh noise changes
        xb, _ = b.round(k, zb, eps)
    tasks = sch.round_tasks(cfg, k_end)
    for t, u, v in zip(tasks, xa, xb):
        same = np.allclose(u, v, atol=1e-12)
        # only the stage-0 task (the perturbed chunk itself) may differ
        assert same == (t.stage != 0), (t.stage, same)


def test_sharp_model_tolerance_separates_rounding_from_a_mask_mistake():
    """The GPU parity bars of the sharp DiT test (weights ~ N(0, 0.05)) must
    admit the spread that bf16 rounding alone causes and reject a planted
    mistake: queries that also see noisier live chunks (the reverse edges
    the WF mask removes, Sec. 3.1)."""
    from gpu_helpers import scaled_errors
    import oracle.dit as od

    cfg = sch.Cfg(S=2, n_chunks=6, history=1)
    dims = dit.Dims(dim=256, heads=2, head_dim=128, ffn=512, layers=2, channels=16, freq=256)
    grid = (3, 8, 10)
    params = wf_synth.dit_params(12, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                 std=0.05)

    def run(b16):
        m = dit.Model(cfg, grid, dims, dit.weights_from(params), [1000.0, 500.0], bf16_points=b16)
        outs = []
        for k in range(sch.n_rounds(cfg)):
            z = lat(12, k, -1, dims, grid)
            outs += m.round(k, z, [lat(12, k - s, s, dims, grid) for s in range(2)])[0]
        return outs

    def worst(a, b):
        w = [0.0, 0.0, 0.0]
        for u, v in zip(a, b):
            w = [max(p, q) for p, q in zip(w, scaled_errors(u, v))]
        return w

    ref = run(True)
    noise = worst(ref, run(False))
    orig = od.masked_attention
    try:
        od.masked_attention = lambda q, k, v, mask: orig(q, k, v, np.ones_like(mask))
        bad = worst(ref, run(True))
    finally:
        od.masked_attention = orig
    bars = (5e-2, 4e-3, 1e-2)          # SHARP_MAX, SHARP_MEAN, SHARP_REL of tests/test_gpu_dit.py
    assert all(n <= b / 1.5 for n, b in zip(noise, bars)), noise
    assert all(e >= 3 * b for e, b in zip(bad, bars)), bad


def test_row_quantisation_e4m3():
    """Per-row e4m3 weights: the row maximum maps to 448 exactly, each entry
    is within half an e4m3 step of the original (relative 2^-4 above the
    subnormal range), and an all-zero row stays zero."""
    rng = np.random.default_rng(3)
    w = (rng.normal(size=(6, 40)) * 0.02).astype(np.float32)
    w[2] = 0.0
    q = dit.quantize_rows_e4m3(w)
    sc = np.abs(w).max(axis=1, keepdims=True).astype(np.float64) / 448.0
    for n in (0, 1, 3, 4, 5):
        i = np.argmax(np.abs(w[n]))
        assert np.isclose(abs(q[n, i]), abs(float(w[n, i])), rtol=1e-6)
    big = np.abs(w) >= 2.0 ** -6 * sc
    assert np.all(np.abs(q - w)[big] <= 2.0 ** -4 * np.abs(w)[big] * (1 + 1e-6))
    assert np.all(q[2] == 0.0)


def test_linear_fp8_model_runs_and_stays_close():
    """The e4m3-linear model is the same computation up to e4m3 rounding of
    weights and activations: close to the bf16 model on a small request."""
    cfg = sch.Cfg(S=2, n_chunks=3, history=1)
    dims = dit.Dims(dim=128, heads=1, head_dim=128, ffn=256, layers=1, channels=16, freq=32)
    grid = (3, 2, 3)
    params = wf_synth.dit_params(4, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                 std=0.02)
    a = dit.Model(cfg, grid, dims, dit.weights_from(params), [1000.0, 500.0])
    b = dit.Model(cfg, grid, dims, dit.weights_from(params), [1000.0, 500.0], linear_fp8=True)
    for k in range(sch.n_rounds(cfg)):
        z = lat(4, k, -1, dims, grid)
        eps = [lat(4, k - s, s, dims, grid) for s in range(2)]
        xa, _ = a.round(k, z, eps)
        xb, _ = b.round(k, z, eps)
        for u, v in zip(xa, xb):
            rel = np.linalg.norm(u - v) / np.linalg.norm(u)
            assert 0 < rel < 5e-2, rel
