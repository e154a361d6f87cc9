"""GPU parity of the DiT path through the C ABI against the fp64 oracle
(oracle/dit.py): the QKV projection fused with RoPE and paged publication
(with and without the Wan2.1 q/k RMSNorm),
whole wavefront rounds of the chunk-wise causal DiT over a request (fill,
steady state with anchor re-rotation, drain), and the Wan2.1-1.3B-shaped
linear layers on sampled rows.

Tolerances: the oracle rounds to bf16 where the BF16 execution stores a
tensor, so the remaining differences are fp32-vs-fp64 arithmetic, rounding
ties and the bf16 softmax probabilities of the attention kernel.  Outputs are
compared as O / max(1, |O|).  The benchmark's random-init model (weights
~ N(0, 0.02)) is held to the stated bf16 bars (max-abs 2e-2, mean-abs 2e-3,
relative L2 2e-2).  The sharper model (weights ~ N(0, 0.05): near one-hot
softmax rows, O(1) gates) amplifies any rounding difference through layers
and rounds; its bars (max 5e-2, mean 4e-3, relative L2 1e-2) are set from the
oracle's own bf16-vs-fp64 spread and checked on the CPU to sit far below the
error of a planted mask mistake (tests/test_oracle_dit.py)."""

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
import wf_synth
from gpu_helpers import scaled_errors
from oracle import dit
from oracle import rope as orope
from oracle import schedule as sch

pytestmark = pytest.mark.gpu

MAX, MEAN, REL = 2e-2, 2e-3, 2e-2
SHARP_STD = 0.05
SHARP_MAX, SHARP_MEAN, SHARP_REL = 5e-2, 4e-3, 1e-2


def new_round(cfg, grid, heads, layers, fp8=None):
    return wf.Round(cfg.S, grid[0] * grid[1] * grid[2], heads, 128, cfg.history,
                    n_chunks=cfg.n_chunks, layers=layers, grid=grid,
                    dtype=wf.WF_FP8 if fp8 else wf.WF_BF16, fp8_scales=fp8 or (1.0, 1.0),
                    use_anchor=cfg.use_anchor, anchor_mode=cfg.anchor_mode, mask=cfg.mask,
                    store_extra=cfg.store_extra,
                    schedule=wf.WF_SCHED_SEQUENTIAL if cfg.sequential else wf.WF_SCHED_WAVEFRONT)


# ---- QKV projection + RoPE + publication -------------------------------------------

def test_qkv_projection_publish_matches_oracle():
    """Q in the query workspace, K/V in the task's page, the anchor's
    unrotated key and its re-rotation (App. B.3), over every round of a
    request whose window shifts."""
    cfg = sch.Cfg(4, 10, 3)
    grid, H = (3, 10, 10), 2
    NC, dim = 300, 256
    r = new_round(cfg, grid, H, 1)
    w = wf_synth.normal(wf_synth.key_of(31, 1), (3 * dim, dim), 0.05, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(31, 2), (3 * dim,), 0.5, torch.bfloat16)
    wd, bd = w.cuda(), b.cuda()
    W, Bv = w.double().numpy(), b.double().numpy()
    P = r.pool_view()
    ys = {}

    def x_of(c, s):
        return wf_synth.normal(wf_synth.key_of(31, 3, c, s), (NC, dim), 1.0, torch.bfloat16)

    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        x = torch.zeros((cfg.S + 1, NC, dim), dtype=torch.bfloat16)
        for i in range(info.n_tasks):
            x[info.task_stage[i]] = x_of(info.task_chunk[i], info.task_stage[i])
        r.publish_proj(0, x.cuda(), wd, bd)
        torch.cuda.synchronize()
        qb = r.qbuf.view(cfg.S + 1, H, NC, 128)
        for t in sch.round_tasks(cfg, k):
            y = x_of(t.chunk, t.stage).double().numpy() @ W.T + Bv
            q, kk, v = (y[:, i * dim:(i + 1) * dim].reshape(NC, H, 128) for i in range(3))
            ys[(t.chunk, t.stage)] = kk
            vg = P[t.dest_page, 0, 1].transpose(0, 1).double().cpu().numpy()
            assert np.all(np.abs(vg - v) <= 2 ** -8 * np.abs(v) + 1e-5), (k, t.stage)
            for got, ref in ((qb[t.stage].transpose(0, 1), orope.rope_chunk(q, t.chunk, grid, 1e4)),
                             (P[t.dest_page, 0, 0].transpose(0, 1),
                              orope.rope_chunk(kk, t.chunk, grid, 1e4))):
                g = got.double().cpu().numpy()
                assert np.all(np.abs(g - ref) <= 2 ** -7 * np.abs(ref) + 1e-4), (k, t.stage)
        if sch.anchor_present(cfg, k):
            raw = ys[(0, cfg.S)]
            rg = P[sch.raw_anchor_page(cfg), 0, 0].transpose(0, 1).double().cpu().numpy()
            assert np.all(np.abs(rg - raw) <= 2 ** -8 * np.abs(raw) + 1e-5)
            # re-rotated from the bf16 unrotated copy (or, before the window
            # first moves, rotated from the fp32 projection): both within bf16
            # rounding of the pair's norm of the exact rotation
            aref = orope.rope_chunk(raw, sch.anchor_tpos(cfg, k), grid, 1e4)
            pair = np.repeat(np.hypot(aref[..., 0::2], aref[..., 1::2]), 2, axis=-1)
            ag = P[0, 0, 0].transpose(0, 1).double().cpu().numpy()
            assert np.all(np.abs(ag - aref) <= 2 ** -7 * pair + 1e-4), k
    assert r.sync_status() == wf.WF_OK


def _norm_ref(x, W, Bv, nq, nk, dim, H):
    """Projection, bf16 rounding of q | k (the stored projection output), the
    q/k RMSNorm over the full width, as the oracle computes them: (q, k, v)
    [rows, H, 128] before RoPE."""
    y = x @ W.T + Bv
    q = dit.rms_norm(dit.bf16(y[:, :dim]), nq)
    k = dit.rms_norm(dit.bf16(y[:, dim:2 * dim]), nk)
    return (a.reshape(len(x), H, 128) for a in (q, k, y[:, 2 * dim:]))


def _pair_close(got, ref, rel=2 ** -7, atol=1e-4):
    """Within rel of each rotary pair's norm: RoPE mixes a pair, so one
    rounding step of an input moves both members by up to that step."""
    pair = np.repeat(np.hypot(ref[..., 0::2], ref[..., 1::2]), 2, axis=-1)
    return np.all(np.abs(got - ref) <= rel * pair + atol)


@pytest.mark.parametrize("fp8", [None, (4.0, 2.0)], ids=["bf16", "e4m3"])
def test_qkv_projection_norm_publish_matches_oracle(fp8):
    """The projection with the Wan2.1 q/k RMSNorm (App. D.2): Q and K
    normalised over the full width before RoPE, V untouched, the anchor's
    normalised unrotated key and its re-rotation, every round of a request
    whose window shifts; bf16 and e4m3 pages."""
    cfg = sch.Cfg(4, 10, 3)
    grid, H = (3, 10, 10), 2
    NC, dim = 300, 256
    r = new_round(cfg, grid, H, 1, fp8)
    w = wf_synth.normal(wf_synth.key_of(35, 1), (3 * dim, dim), 0.05, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(35, 2), (3 * dim,), 0.5, torch.bfloat16)
    nq = (1 + wf_synth.normal(wf_synth.key_of(35, 4), (dim,), 0.3)).to(torch.bfloat16)
    nk = (1 + wf_synth.normal(wf_synth.key_of(35, 5), (dim,), 0.3)).to(torch.bfloat16)
    W, Bv = w.double().numpy(), b.double().numpy()
    NQ, NK = nq.double().numpy(), nk.double().numpy()
    P = r.pool_view()
    sq, sv = fp8 or (1.0, 1.0)
    # bf16: the fp32 projection may round to a bf16 value one ulp away from
    # the fp64 one (up to 2^-7 of that element, spread over its rotary pair
    # by RoPE) before the norm, and the result is rounded again (up to 2^-8):
    # 2^-6 of the pair norm covers both; e4m3: one e4m3 step (2^-3
    # relative) or the subnormal step 2^-9 near zero.  The norm kernel alone
    # is checked more tightly below, from the GPU's own projection output.
    rel, vrel = (2 ** -3, 2 ** -3) if fp8 else (2 ** -6, 2 ** -8)
    atol = 2 ** -9 / sq if fp8 else 1e-4
    vatol = 2 ** -9 / sv if fp8 else 1e-5
    dimq = dim
    raws = {}

    def x_of(c, s):
        return wf_synth.normal(wf_synth.key_of(35, 3, c, s), (NC, dim), 1.0, torch.bfloat16)

    def page(t):
        return t.float().cpu().double().numpy()

    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        x = torch.zeros((cfg.S + 1, NC, dim), dtype=torch.bfloat16)
        for i in range(info.n_tasks):
            x[info.task_stage[i]] = x_of(info.task_chunk[i], info.task_stage[i])
        r.publish_proj(0, x.cuda(), w.cuda(), b.cuda(), nq.cuda(), nk.cuda())
        torch.cuda.synchronize()
        qb = r.qbuf.view(cfg.S + 1, H, NC, 128)
        # the norm kernel from the bf16 q | k rows the projection left: the
        # same input as the kernel's, so only the final rounding remains
        # (half an output ulp, <= 2^-8 of the pair norm) for bf16 pages
        lin = r._qk_tmp.view(torch.bfloat16).view(cfg.S + 1, NC, 2 * dim).double().cpu().numpy()
        for t in sch.round_tasks(cfg, k):
            if fp8:
                break
            qe = dit.rms_norm(lin[t.stage, :, :dimq], NQ).reshape(NC, H, 128)
            ke = dit.rms_norm(lin[t.stage, :, dimq:], NK).reshape(NC, H, 128)
            for got, ref in ((qb[t.stage], qe), (P[t.dest_page, 0, 0], ke)):
                assert _pair_close(page(got.transpose(0, 1)), orope.rope_chunk(ref, t.chunk, grid, 1e4),
                                   2 ** -8 * (1 + 1e-4), 1e-6), (k, t.stage)
        for t in sch.round_tasks(cfg, k):
            q, kk, v = _norm_ref(x_of(t.chunk, t.stage).double().numpy(), W, Bv, NQ, NK, dim, H)
            raws[(t.chunk, t.stage)] = kk
            vg = page(P[t.dest_page, 0, 1].transpose(0, 1)) / sv
            assert np.all(np.abs(vg - v) <= vrel * np.abs(v) + vatol), (k, t.stage)
            assert _pair_close(page(qb[t.stage].transpose(0, 1)) / sq,
                               orope.rope_chunk(q, t.chunk, grid, 1e4), rel, atol), (k, t.stage)
            assert _pair_close(page(P[t.dest_page, 0, 0].transpose(0, 1)) / sq,
                               orope.rope_chunk(kk, t.chunk, grid, 1e4), rel, atol), (k, t.stage)
        if sch.anchor_present(cfg, k):
            raw = raws[(0, cfg.S)]
            rg = page(P[sch.raw_anchor_page(cfg), 0, 0].transpose(0, 1)) / sq
            assert np.all(np.abs(rg - raw) <= rel * np.abs(raw) + atol), k
            # re-rotated from the rounded unrotated copy: two roundings
            aref = orope.rope_chunk(raw, sch.anchor_tpos(cfg, k), grid, 1e4)
            ag = page(P[0, 0, 0].transpose(0, 1)) / sq
            assert _pair_close(ag, aref, 2 * rel, 2 * atol), k
    assert r.sync_status() == wf.WF_OK


def test_qkv_projection_rejects_half_a_norm():
    cfg = sch.Cfg(2, 4, 1)
    r = new_round(cfg, (3, 4, 4), 2, 1)
    r.step()
    x = torch.zeros((3, 48, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((768, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr() if t is not None else None
    fn = wf.lib.wf_qkv_proj_rope_publish
    assert fn(r.plan, 0, p(x), p(w), None, p(g), None, p(x), None) == wf.WF_EINVAL
    assert fn(r.plan, 0, p(x), p(w), None, p(g), p(g), None, None) == wf.WF_EINVAL
    torch.cuda.synchronize()


# ---- whole rounds ---------------------------------------------------------------------

def run_request(cfg, grid, heads, dims, std, seed, steps, fp8=None, linear_fp8=False):
    params = wf_synth.dit_params(seed, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                 std=std)
    oracle = dit.Model(cfg, grid, dims, dit.weights_from(params), steps, bf16_points=True,
                       kv_fp8=fp8, linear_fp8=linear_fp8)
    r = new_round(cfg, grid, heads, dims.layers, fp8)
    model = wf.Dit(r, params, ffn=dims.ffn, channels=dims.channels, freq=dims.freq,
                   timesteps=steps, linear_fp8=linear_fp8)
    C, F, Hl, Wl = dims.channels, grid[0], 2 * grid[1], 2 * grid[2]
    latent = C * F * Hl * Wl
    worst = [0.0, 0.0, 0.0]
    n_emitted = 0
    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        z = wf_synth.latent(seed, k, -1, C, F, Hl, Wl)
        eps = torch.stack([wf_synth.latent(seed, k - s, s, C, F, Hl, Wl) for s in range(cfg.S)])
        x0 = torch.full((cfg.S + 1, latent), float("nan"), device="cuda")
        out = torch.full((latent,), float("nan"), device="cuda")
        model.round(z.cuda(), eps.cuda(), x0, out)
        torch.cuda.synchronize()
        ref_x0, ref_out = oracle.round(k, z.double().numpy(),
                                       [e.double().numpy() for e in eps])
        for t, ref in zip(sch.round_tasks(cfg, k), ref_x0):
            got = x0[t.stage].cpu().numpy().reshape(ref.shape)
            e = scaled_errors(got, ref)
            worst = [max(a, b) for a, b in zip(worst, e)]
        if ref_out is not None:
            got = out.cpu().numpy().reshape(ref_out.shape)
            e = scaled_errors(got, ref_out)
            worst = [max(a, b) for a, b in zip(worst, e)]
            n_emitted += 1
        else:
            assert torch.isnan(out).all()      # nothing finished this round: untouched
    assert r.sync_status() == wf.WF_OK
    assert n_emitted == cfg.n_chunks
    r.close()
    return worst


DIMS = dit.Dims(dim=256, heads=2, head_dim=128, ffn=512, layers=2, channels=16, freq=256)
GRID = (3, 8, 10)       # 240 tokens per chunk: one full 128-row tile and a ragged one


@pytest.mark.parametrize("cfg", [sch.Cfg(2, 6, 1), sch.Cfg(3, 5, -1),
                                 sch.Cfg(2, 5, 2, anchor_mode=sch.ANCHOR_ABSOLUTE),
                                 sch.Cfg(2, 5, 1, mask=sch.MASK_RF),
                                 sch.Cfg(2, 4, 1, sequential=True),
                                 sch.Cfg(2, 6, 1, store_extra=2)], ids=str)
def test_dit_request_matches_oracle(cfg):
    steps = [1000.0, 750.0, 500.0, 250.0][:cfg.S] if cfg.S != 2 else [1000.0, 500.0]
    mx, mean, rel = run_request(cfg, GRID, DIMS.heads, DIMS, std=SHARP_STD, seed=12, steps=steps)
    assert mx <= SHARP_MAX and mean <= SHARP_MEAN and rel <= SHARP_REL, (mx, mean, rel)


def test_dit_request_baseline_init():
    """Weights ~ N(0, 0.02) as in the benchmark's random-init model."""
    cfg = sch.Cfg(4, 6, 3)
    mx, mean, rel = run_request(cfg, GRID, DIMS.heads, DIMS, std=0.02, seed=13,
                                steps=[1000.0, 750.0, 500.0, 250.0])
    assert mx <= MAX and mean <= MEAN and rel <= REL, (mx, mean, rel)


def test_dit_request_five_steps():
    """The 5-step schedule of App. A (S = 5: six tasks per round, contexts of
    up to ten chunks with W = 3) over a whole request with eviction."""
    cfg = sch.Cfg(5, 9, 3)
    mx, mean, rel = run_request(cfg, GRID, DIMS.heads, DIMS, std=0.02, seed=16,
                                steps=[1000.0, 800.0, 600.0, 400.0, 200.0])
    assert mx <= MAX and mean <= MEAN and rel <= REL, (mx, mean, rel)


def test_dit_request_wan_width():
    """The Wan2.1-1.3B block width (dim 1536, 12 heads x 128, FFN 8960) on a
    small grid (3 x 8 x 10 patches), two blocks, the benchmark's weights
    ~ N(0, 0.02): the LayerNorm, QKV epilogue, q/k RMSNorm and attention
    paths of the benchmarked model.  At this width the bf16 rounding points
    alone move the oracle's predictions by max 0.014, mean 0.0023, relative
    L2 0.0039 (bf16 vs fp64 oracle, tests/derive_wan_width_bars.py), above
    the 2e-3 mean bar, so the bars are the sharp model's (5e-2, 4e-3, 1e-2);
    a planted mask mistake moves them by 0.28 / 0.056 / 0.097."""
    cfg = sch.Cfg(4, 6, 3)
    dims = dit.Dims(dim=1536, heads=12, head_dim=128, ffn=8960, layers=2, channels=16, freq=256)
    mx, mean, rel = run_request(cfg, GRID, dims.heads, dims, std=0.02, seed=18,
                                steps=[1000.0, 750.0, 500.0, 250.0])
    assert mx <= SHARP_MAX and mean <= SHARP_MEAN and rel <= SHARP_REL, (mx, mean, rel)


def test_dit_round_deterministic():
    cfg = sch.Cfg(2, 4, 1)
    dims = DIMS
    params = wf_synth.dit_params(14, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                 std=0.1)
    outs = []
    for _ in range(2):
        r = new_round(cfg, GRID, dims.heads, dims.layers)
        m = wf.Dit(r, params, ffn=dims.ffn, timesteps=[1000.0, 500.0])
        lat = 16 * 3 * 16 * 20
        got = []
        for k in range(sch.n_rounds(cfg)):
            r.step()
            z = wf_synth.latent(14, k, -1, 16, 3, 16, 20).cuda()
            eps = torch.stack([wf_synth.latent(14, k - s, s, 16, 3, 16, 20) for s in range(2)]).cuda()
            x0 = torch.zeros((3, lat), device="cuda")
            m.round(z, eps, x0)
            got.append(x0.clone())
        torch.cuda.synchronize()
        outs.append(torch.stack(got))
        r.close()
    assert torch.equal(outs[0], outs[1])


# ---- Wan2.1-1.3B shapes, sampled rows ---------------------------------------------------

def test_wan13_linears_sampled_rows():
    """The four GEMM shapes of one Wan2.1-1.3B block over a steady round
    (T = 5 x 4680 rows): QKV 1536 -> 4608, output 1536 -> 1536, FFN 1536 ->
    8960 (GELU) and 8960 -> 1536 (gated residual), checked on sampled rows."""
    T, dim, ffn = 5 * 4680, 1536, 8960
    r = wf.Round(1, 48, 1, 128, -1, n_chunks=1, grid=(3, 4, 4), dtype=wf.WF_BF16)
    rows = np.array([0, 1, 127, 128, 4679, 4680, 9000, 23271, 23272, 23399])
    for (N, K, epi, seed) in ((3 * dim, dim, wf.WF_EPI_BF16, 1), (dim, dim, wf.WF_EPI_GATED_RESIDUAL, 2),
                              (ffn, dim, wf.WF_EPI_GELU_BF16, 3), (dim, ffn, wf.WF_EPI_GATED_RESIDUAL, 4)):
        a = wf_synth.normal(wf_synth.key_of(seed, 1), (T, K), 1.0, torch.bfloat16)
        w = wf_synth.normal(wf_synth.key_of(seed, 2), (N, K), 0.02, torch.bfloat16)
        b = wf_synth.normal(wf_synth.key_of(seed, 3), (N,), 0.02, torch.bfloat16)
        y = a[rows].double().numpy() @ w.double().numpy().T + b.double().numpy()
        if epi == wf.WF_EPI_GATED_RESIDUAL:
            gate = wf_synth.normal(wf_synth.key_of(seed, 4), (5, N), 1.0, torch.float32)
            x = wf_synth.normal(wf_synth.key_of(seed, 5), (T, N), 1.0, torch.float32)
            out = x.cuda()
            r.linear(a.cuda(), w.cuda(), b.cuda(), out, epi, gate=gate.cuda(), rows_per_group=4680)
            ref = x[rows].double().numpy() + gate.double().numpy()[rows // 4680] * y
            got = out[torch.from_numpy(rows).cuda()].cpu().double().numpy()
            assert np.abs(got - ref).max() <= 1e-3, (N, K)
        else:
            out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
            r.linear(a.cuda(), w.cuda(), b.cuda(), out, epi)
            ref = dit.gelu_tanh(y) if epi == wf.WF_EPI_GELU_BF16 else y
            got = out[torch.from_numpy(rows).cuda()].cpu().double().numpy()
            assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-4), (N, K)
        torch.cuda.synchronize()
        del a, w, out
    assert r.sync_status() == wf.WF_OK
    r.close()


@pytest.mark.parametrize("width", ["wan13", "wan13-norm", "14b-norm"])
def test_qkv_publish_sampled_rows(width):
    """The fused QKV projection + RoPE + paged publication at full size in a
    steady round -- Wan2.1-1.3B (dim 1536 -> 4608, 12 heads), with and
    without the q/k RMSNorm, and the 14B width (dim 5120 -> 15360, 40 heads)
    with it -- 5 tasks of 4680 tokens, checked on sampled tokens of every
    task against the fp64 oracle."""
    cfg = sch.Cfg(4, 14, 3)
    grid = (3, 30, 52)
    H = 40 if width == "14b-norm" else 12
    NC, dim = 4680, 128 * H
    norm = width.endswith("norm")
    r = new_round(cfg, grid, H, 1)
    w = wf_synth.normal(wf_synth.key_of(41, 1), (3 * dim, dim), 0.02, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(41, 2), (3 * dim,), 0.02, torch.bfloat16)
    nq = (1 + wf_synth.normal(wf_synth.key_of(41, 4), (dim,), 0.02)).to(torch.bfloat16)
    nk = (1 + wf_synth.normal(wf_synth.key_of(41, 5), (dim,), 0.02)).to(torch.bfloat16)
    W, Bv = w.double().numpy(), b.double().numpy()
    wd, bd = w.cuda(), b.cuda()
    nqd, nkd = (nq.cuda(), nk.cuda()) if norm else (None, None)
    rows = np.array([0, 1, 127, 128, 2500, 4607, 4608, 4679])
    k_check = cfg.S + cfg.history + 2
    xs = {}
    for k in range(k_check + 1):
        info = r.step()
        x = torch.empty((cfg.S + 1, NC, dim), dtype=torch.bfloat16)
        for i in range(info.n_tasks):
            c, s_ = info.task_chunk[i], info.task_stage[i]
            xs[(c, s_)] = wf_synth.normal(wf_synth.key_of(41, 3, c, s_), (NC, dim), 1.0, torch.bfloat16)
            x[s_] = xs[(c, s_)]
        r.publish_proj(0, x.cuda(), wd, bd, nqd, nkd)
        del x
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_OK
    P = r.pool_view()
    qb = r.qbuf.view(cfg.S + 1, H, NC, 128)
    t_idx = torch.from_numpy(rows).cuda()
    for t in sch.round_tasks(cfg, k_check):
        xr = xs[(t.chunk, t.stage)][rows].double().numpy()
        if norm:
            q, kk, v = _norm_ref(xr, W, Bv, nq.double().numpy(), nk.double().numpy(), dim, H)
        else:
            y = xr @ W.T + Bv
            q, kk, v = (y[:, i * dim:(i + 1) * dim].reshape(len(rows), H, 128) for i in range(3))
        # RoPE of the sampled tokens at their (t, h, w) positions
        pos = [p[rows] for p in orope.chunk_positions(t.chunk, *grid)]
        ang = orope.pair_angles(128, 1e4, *pos)
        qr, kr = orope.rotate(q, ang), orope.rotate(kk, ang)
        got_q = qb[t.stage][:, t_idx].transpose(0, 1).double().cpu().numpy()
        got_k = P[t.dest_page, 0, 0][:, t_idx].transpose(0, 1).double().cpu().numpy()
        got_v = P[t.dest_page, 0, 1][:, t_idx].transpose(0, 1).double().cpu().numpy()
        # with the norm, a one-ulp difference of the bf16 projection output
        # the norm reads (fp32 vs fp64 accumulation) joins the final rounding
        for g, ref in ((got_q, qr), (got_k, kr)):
            assert _pair_close(g, ref, 2 ** -6 if norm else 2 ** -7, 1e-3), t.stage
        assert np.all(np.abs(got_v - v) <= 2 ** -7 * np.abs(v) + 1e-3), t.stage
    r.close()



# ---- 8-bit attention inside the DiT round ------------------------------------------

# 8-bit bars (tests/derive_fp8_bars.py).  Benchmark weights (std 0.02): the
# emulated e4m3 rounding of P moves the predictions by max <= 0.0064, so max
# 0.05 (a mask mistake at this flat attention moves them by only ~0.025:
# the sharp variant below is the one that separates mistakes).  Sharp
# weights (std 0.05): rounding spread max 0.094 / mean 0.011 / rel 0.017
# (e4m3 linears and attention), planted mask mistake 0.46 / 0.071 / 0.117.
FP8_REL, FP8_MEAN, FP8_MAX = 4e-2, 1.5e-2, 5e-2
FP8_SHARP = (0.15, 0.02, 0.035)


@pytest.mark.parametrize("std", [0.02, 0.05], ids=["bench-init", "sharp"])
def test_dit_request_fp8_attention(std):
    """A WF_FP8 plan runs the same DiT round with e4m3 Q/K/V pages (written by
    the QKV epilogue) and e4m3 attention; checked against the oracle with
    the same e4m3 storage."""
    cfg = sch.Cfg(4, 6, 3)
    mx, mean, rel = run_request(cfg, GRID, DIMS.heads, DIMS, std=std, seed=13,
                                steps=[1000.0, 750.0, 500.0, 250.0], fp8=(4.0, 4.0))
    bars = (FP8_MAX, FP8_MEAN, FP8_REL) if std == 0.02 else FP8_SHARP
    assert mx <= bars[0] and mean <= bars[1] and rel <= bars[2], (mx, mean, rel)


def test_qkv_projection_publish_fp8():
    """The QKV epilogue's e4m3 pages: V, K and Q (after RoPE) within one e4m3
    step of the oracle (fp32 vs fp64 before the rounding), the anchor's
    unrotated key likewise."""
    cfg = sch.Cfg(3, 7, 2)
    grid, H = (3, 10, 10), 2
    NC, dim = 300, 256
    scales = (4.0, 2.0)
    r = new_round(cfg, grid, H, 1, fp8=scales)
    w = wf_synth.normal(wf_synth.key_of(33, 1), (3 * dim, dim), 0.05, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(33, 2), (3 * dim,), 0.5, torch.bfloat16)
    W, Bv = w.double().numpy(), b.double().numpy()
    P = r.pool_view()
    ys = {}

    def x_of(c, s):
        return wf_synth.normal(wf_synth.key_of(33, 3, c, s), (NC, dim), 1.0, torch.bfloat16)

    def close(got, ref, scale):
        g = got.float().cpu().double().numpy() / scale
        return np.all(np.abs(g - ref) <= 2 ** -3 * np.abs(ref) + 2 ** -9 / scale)

    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        x = torch.zeros((cfg.S + 1, NC, dim), dtype=torch.bfloat16)
        for i in range(info.n_tasks):
            x[info.task_stage[i]] = x_of(info.task_chunk[i], info.task_stage[i])
        r.publish_proj(0, x.cuda(), w.cuda(), b.cuda())
        torch.cuda.synchronize()
        qb = r.qbuf.view(cfg.S + 1, H, NC, 128)
        for t in sch.round_tasks(cfg, k):
            y = x_of(t.chunk, t.stage).double().numpy() @ W.T + Bv
            q, kk, v = (y[:, i * dim:(i + 1) * dim].reshape(NC, H, 128) for i in range(3))
            ys[(t.chunk, t.stage)] = kk
            assert close(P[t.dest_page, 0, 1].transpose(0, 1), v, scales[1]), (k, t.stage)
            assert close(P[t.dest_page, 0, 0].transpose(0, 1), orope.rope_chunk(kk, t.chunk, grid, 1e4), scales[0])
            assert close(qb[t.stage].transpose(0, 1), orope.rope_chunk(q, t.chunk, grid, 1e4), scales[0])
        if sch.anchor_present(cfg, k):
            assert close(P[sch.raw_anchor_page(cfg), 0, 0].transpose(0, 1), ys[(0, cfg.S)], scales[0])
    assert r.sync_status() == wf.WF_OK
    r.close()



@pytest.mark.parametrize("std", [0.02, 0.05], ids=["bench-init", "sharp"])
@pytest.mark.parametrize("fp8", [None, (4.0, 4.0)], ids=["bf16-attention", "e4m3-attention"])
def test_dit_request_e4m3_linears(fp8, std):
    """The block's linear layers in e4m3 (per-channel weight scales, e4m3 LN
    output, attention output and FFN hidden layer), with bf16 or e4m3
    attention, against the oracle with the same e4m3 rounding points."""
    cfg = sch.Cfg(4, 6, 3)
    mx, mean, rel = run_request(cfg, GRID, DIMS.heads, DIMS, std=std, seed=15,
                                steps=[1000.0, 750.0, 500.0, 250.0], fp8=fp8, linear_fp8=True)
    bars = (FP8_MAX, FP8_MEAN, FP8_REL) if std == 0.02 else FP8_SHARP
    assert mx <= bars[0] and mean <= bars[1] and rel <= bars[2], (mx, mean, rel)
