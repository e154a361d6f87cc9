"""GPU parity of whole DiT rounds over a group of requests
(wf_group_dit_bind / wf_group_dit_round).

"Wave Forcing" names serving concurrent streams with batching as the next
step (Sec. 8 Future Work; App. E).  A group DiT round runs the chunk-wise
causal DiT forward of Sec. 2 Eq. 1 / Sec. 4.1 Eq. 8-9 for the tasks of every
selected member in one pass.  Members start at different rounds and one
pauses for a round, so the batched rounds mix fill, steady state and drain
and the members' round parities differ.  Checked: every member's
predictions and emitted chunks against the fp64 oracle of its own request
(the bars of tests/test_gpu_dit.py for the sharp model), and bit-identity
with the member's own single-plan wf_dit_round (same kernels, the rows only
moved), in bf16 and with 8-bit attention and linear layers."""

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
import wf_synth
from gpu_helpers import scaled_errors
from oracle import dit
from oracle import schedule as sch

pytestmark = pytest.mark.gpu

SHARP_MAX, SHARP_MEAN, SHARP_REL = 5e-2, 4e-3, 1e-2
DIMS = dit.Dims(dim=256, heads=2, head_dim=128, ffn=512, layers=2, channels=16, freq=256)
GRID = (3, 8, 10)       # 240 tokens per chunk: one full 128-row tile and a ragged one
C, F, HL, WL = 16, 3, 16, 20
LATENT = C * F * HL * WL


def _kw(cfg, fp8):
    return dict(n_chunks=cfg.n_chunks, layers=DIMS.layers, grid=GRID,
                dtype=wf.WF_FP8 if fp8 else wf.WF_BF16, fp8_scales=fp8 or (1.0, 1.0),
                use_anchor=cfg.use_anchor, anchor_mode=cfg.anchor_mode, mask=cfg.mask,
                store_extra=cfg.store_extra)


def _inputs(seed, r, k, S):
    z = wf_synth.latent(seed + 97 * r, k, -1, C, F, HL, WL)
    eps = torch.stack([wf_synth.latent(seed + 97 * r, k - s, s, C, F, HL, WL) for s in range(S)])
    return z, eps


def run_group(cfg, starts, pause, params, steps, seed, fp8=None, linear_fp8=False):
    """Drive the members (member r from global round starts[r]; member
    pause[0] skips global round pause[1]) with group DiT rounds; returns per
    member the list of (k, {stage: x0}, chunk or None)."""
    n = len(starts)
    grp = wf.Group(n, cfg.S, GRID[0] * GRID[1] * GRID[2], DIMS.heads, 128, cfg.history,
                   **_kw(cfg, fp8))
    model = wf.GroupDit(grp, params, ffn=DIMS.ffn, channels=C, freq=DIMS.freq, timesteps=steps,
                        linear_fp8=linear_fp8)
    res = [[] for _ in range(n)]
    done = [False] * n
    g = 0
    while not all(done):
        mask, infos = 0, {}
        for r in range(n):
            if g < starts[r] or done[r] or (r, g) == pause:
                continue
            info = grp.rounds[r].step()
            if info is None:
                done[r] = True
                continue
            infos[r] = info
            mask |= 1 << r
        g += 1
        if not mask:
            continue
        z = torch.zeros((n, LATENT))
        eps = torch.zeros((n, cfg.S, LATENT))
        for r, info in infos.items():
            zr, er = _inputs(seed, r, info.k, cfg.S)
            z[r], eps[r] = zr.reshape(-1), er.reshape(cfg.S, -1)
        x0 = torch.full((n, cfg.S + 1, LATENT), float("nan"), device="cuda")
        out = torch.full((n, LATENT), float("nan"), device="cuda")
        model.round(mask, z.cuda(), eps.cuda(), x0, out)
        torch.cuda.synchronize()
        for r, info in infos.items():
            stages = [info.task_stage[i] for i in range(info.n_tasks)]
            o = out[r].cpu()
            res[r].append((info.k, {s: x0[r, s].cpu() for s in stages},
                           None if torch.isnan(o).all() else o))
    assert grp.rounds[0].sync_status() == wf.WF_OK
    grp.close()
    return res


def run_single(cfg, r_id, params, steps, seed, fp8=None, linear_fp8=False):
    rnd = wf.Round(cfg.S, GRID[0] * GRID[1] * GRID[2], DIMS.heads, 128, cfg.history, **_kw(cfg, fp8))
    model = wf.Dit(rnd, params, ffn=DIMS.ffn, channels=C, freq=DIMS.freq, timesteps=steps,
                   linear_fp8=linear_fp8)
    res = []
    for k in range(sch.n_rounds(cfg)):
        info = rnd.step()
        z, eps = _inputs(seed, r_id, k, cfg.S)
        x0 = torch.full((cfg.S + 1, LATENT), float("nan"), device="cuda")
        out = torch.full((LATENT,), float("nan"), device="cuda")
        model.round(z.cuda(), eps.cuda(), x0, out)
        torch.cuda.synchronize()
        stages = [info.task_stage[i] for i in range(info.n_tasks)]
        o = out.cpu()
        res.append((k, {s: x0[s].cpu() for s in stages}, None if torch.isnan(o).all() else o))
    assert rnd.sync_status() == wf.WF_OK
    rnd.close()
    return res


@pytest.mark.parametrize("fp8,linear_fp8", [(None, False), ((4.0, 2.0), False), ((4.0, 2.0), True)],
                         ids=["bf16", "e4m3-attention", "w8a8"])
def test_group_dit_bit_identical_to_single_plans(fp8, linear_fp8):
    cfg = sch.Cfg(3, 5, 1)
    steps = [1000.0, 700.0, 400.0]
    params = wf_synth.dit_params(41, DIMS.dim, DIMS.ffn, DIMS.layers, C, DIMS.freq, std=0.05)
    starts, pause = [0, 1, 3], (1, 4)
    got = run_group(cfg, starts, pause, params, steps, 41, fp8, linear_fp8)
    for r in range(len(starts)):
        want = run_single(cfg, r, params, steps, 41, fp8, linear_fp8)
        assert len(got[r]) == len(want) == sch.n_rounds(cfg)
        for (kg, xg, og), (kw, xw, ow) in zip(got[r], want):
            assert kg == kw and xg.keys() == xw.keys()
            for s in xw:
                assert torch.equal(xg[s], xw[s]), (r, kw, s)
            assert (og is None) == (ow is None), (r, kw)
            if ow is not None:
                assert torch.equal(og, ow), (r, kw)


@pytest.mark.parametrize("cfg", [sch.Cfg(2, 5, 1), sch.Cfg(3, 4, -1, mask=sch.MASK_RF)], ids=str)
def test_group_dit_matches_oracle(cfg):
    steps = [1000.0, 500.0] if cfg.S == 2 else [1000.0, 700.0, 400.0]
    seed = 43
    params = wf_synth.dit_params(seed, DIMS.dim, DIMS.ffn, DIMS.layers, C, DIMS.freq, std=0.05)
    starts = [0, 2]
    got = run_group(cfg, starts, (0, 3), params, steps, seed)
    for r in range(len(starts)):
        oracle = dit.Model(cfg, GRID, DIMS, dit.weights_from(params), steps, bf16_points=True)
        emitted = 0
        for k, x0, out in got[r]:
            z, eps = _inputs(seed, r, k, cfg.S)
            ref_x0, ref_out = oracle.round(k, z.double().numpy(), [e.double().numpy() for e in eps])
            for t, ref in zip(sch.round_tasks(cfg, k), ref_x0):
                mx, mean, rel = scaled_errors(x0[t.stage].numpy().reshape(ref.shape), ref)
                assert mx <= SHARP_MAX and mean <= SHARP_MEAN and rel <= SHARP_REL, (r, k, t.stage)
            assert (out is None) == (ref_out is None), (r, k)
            if ref_out is not None:
                mx, mean, rel = scaled_errors(out.numpy().reshape(ref_out.shape), ref_out)
                assert mx <= SHARP_MAX and mean <= SHARP_MEAN and rel <= SHARP_REL, (r, k)
                emitted += 1
        assert emitted == cfg.n_chunks


def test_group_dit_rejects():
    cfg = sch.Cfg(2, 4, 1)
    grp = wf.Group(2, cfg.S, 240, DIMS.heads, 128, cfg.history, **_kw(cfg, None))
    z = torch.zeros((2, LATENT), device="cuda")
    eps = torch.zeros((2, cfg.S, LATENT), device="cuda")
    fn = wf.lib.wf_group_dit_round
    p = lambda t: t.data_ptr() if t is not None else None
    grp.rounds[0].step()
    assert fn(grp.group, 1, p(z), p(eps), None, None, None) == wf.WF_EUNBOUND
    params = wf_synth.dit_params(44, DIMS.dim, DIMS.ffn, DIMS.layers, C, DIMS.freq, std=0.05)
    model = wf.GroupDit(grp, params, ffn=DIMS.ffn, channels=C, freq=DIMS.freq,
                        timesteps=[1000.0, 500.0])
    assert fn(grp.group, 0, p(z), p(eps), None, None, None) == wf.WF_EINVAL      # empty mask
    assert fn(grp.group, 4, p(z), p(eps), None, None, None) == wf.WF_EINVAL      # bit beyond n
    assert fn(grp.group, 3, p(z), p(eps), None, None, None) == wf.WF_ENOROUND    # member 1 not entered
    assert fn(grp.group, 1, None, p(eps), None, None, None) == wf.WF_EINVAL      # stage 0 needs z_new
    assert fn(grp.group, 1, p(z), None, None, None, None) == wf.WF_EINVAL        # S > 1 needs eps
    model.round(1, z, eps)
    torch.cuda.synchronize()
    assert grp.rounds[0].sync_status() == wf.WF_OK
    grp.close()
