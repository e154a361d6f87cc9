"""GPU parity of 8-bit attention (plan dtype WF_FP8: Q and the K/V pages in
OCP FP8 e4m3, the pages' SageAttention / FP8 K/V axis) against the fp64
oracle with the same e4m3 storage (oracle.round.Fp8).

* Placement: V pages equal the oracle's e4m3 bytes exactly (power-of-two
  scales make the scaling exact); RoPE'd Q and K within one e4m3 step
  (fp32 vs fp64 rotation before the rounding).
* Visibility fingerprint: Q = 0 and V one-hot in {0, 1} are exact in e4m3
  and give P = 1 exactly, so O = 1/|context| per visible entry: masks, pages,
  the e4m3 MMA formats and the TMEM layout of P are checked exactly.
* Whole requests: the remaining difference is the kernel's own e4m3
  rounding of the softmax probabilities P before the PV product (round to
  nearest: up to 2^-4 relative, about 3.6% RMS per element, unbiased), which
  averages over the keys a row attends to.  Sharp inputs (few dominant keys
  per row) measured relative L2 2.4% and mean |O - O_ref| / max(1, |O_ref|)
  0.0076; bars: relative L2 <= 4e-2, mean <= 1.5e-2, max 0.25.  The
  max bar comes from tests/derive_fp8_bars.py: the oracle with that e4m3
  rounding of P emulated differs from the plain oracle by max 0.053-0.074
  on these requests, and a planted mask mistake (reverse edges) by max
  3.7-4.9.  The benchmark's near-uniform rows keep the bf16 bars.  Masks
  and pages are checked exactly by the fingerprint, so the looser bars hide
  no bookkeeping error."""

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
from gpu_helpers import errors, fill_qkv, make_round, raw_fn, scaled_errors
from oracle import rope as orope
from oracle import schedule as sch
from oracle.round import Fp8, Geom, e4m3, round_attention

pytestmark = pytest.mark.gpu

SMALL = Geom(grid_t=3, grid_h=10, grid_w=10, heads=2, head_dim=128)   # 300 tokens: 2 tiles + 44
REL, MEAN, MAX = 4e-2, 1.5e-2, 0.25


def test_fp8_publish_placement():
    cfg = sch.Cfg(4, 10, 3)
    scales = (4.0, 8.0)
    r = make_round(cfg, SMALL, wf.WF_FP8, fp8_scales=scales)
    raw, traw = raw_fn(5, SMALL, torch.bfloat16)
    P = r.pool_view()
    NC, H = SMALL.chunk_tokens, SMALL.heads
    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
        torch.cuda.synchronize()
        qb = r.qbuf.view(cfg.S + 1, H, NC, 128)
        for t in sch.round_tasks(cfg, k):
            x = raw(t.chunk, t.stage, 0)
            # the pages hold the scaled e4m3 values
            vg = P[t.dest_page, 0, 1].transpose(0, 1).float().cpu().double().numpy() / scales[1]
            assert np.array_equal(vg, e4m3(x[:, 2], scales[1]))
            for got, ref in ((qb[t.stage].transpose(0, 1), orope.rope_chunk(x[:, 0], t.chunk, SMALL.grid, 1e4)),
                             (P[t.dest_page, 0, 0].transpose(0, 1), orope.rope_chunk(x[:, 1], t.chunk, SMALL.grid, 1e4))):
                g = got.float().cpu().double().numpy() / scales[0]
                assert np.all(np.abs(g - ref) <= 2 ** -3 * np.abs(ref) + 2 ** -9 / scales[0]), (k, t.stage)
        if sch.anchor_present(cfg, k):
            k0 = raw(0, cfg.S, 0)[:, 1]
            rg = P[sch.raw_anchor_page(cfg), 0, 0].transpose(0, 1).float().cpu().double().numpy()
            assert np.array_equal(rg / scales[0], e4m3(k0, scales[0]))
    assert r.sync_status() == wf.WF_OK
    r.close()


TC_KERNELS = [wf.WF_ATTN_TC]


@pytest.mark.parametrize("kernel", TC_KERNELS)
@pytest.mark.parametrize("cfg", [sch.Cfg(4, 10, 3), sch.Cfg(3, 7, 1, mask=sch.MASK_RF),
                                 sch.Cfg(2, 4, 1, sequential=True), sch.Cfg(1, 4, 1), sch.Cfg(3, 1, -1),
                                 sch.Cfg(3, 7, 0), sch.Cfg(2, 6, 0, use_anchor=False)], ids=str)
def test_fp8_visibility_fingerprint(cfg, kernel):
    geom = SMALL
    r = make_round(cfg, geom, wf.WF_FP8, fp8_scales=(2.0, 1.0))
    out = r.new_out()
    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        qkv = r.new_qkv().zero_()
        for i in range(info.n_tasks):
            c, s = info.task_chunk[i], info.task_stage[i]
            g = torch.Generator().manual_seed(100 * c + s)
            qkv[s, :, 1] = torch.randn(geom.chunk_tokens, geom.heads, geom.head_dim, generator=g).to(torch.bfloat16)
            qkv[s, :, 2, :, c] = 1.0
            qkv[s, :, 2, :, 64 + s] = 1.0
        r.publish(0, qkv)
        r.attention(0, out, kernel)
        torch.cuda.synchronize()
        for t in sch.round_tasks(cfg, k):
            want = np.zeros(geom.head_dim)
            for e in t.context:
                st = e.j if e.kind == sch.KIND_LIVE else cfg.S
                want[e.chunk] += 1.0 / len(t.context)
                want[64 + st] += 1.0 / len(t.context)
            got = out[t.stage].float().cpu().numpy()
            assert np.abs(got - want[None, None, :]).max() <= 2e-3, (k, t.chunk, t.stage)
    assert r.sync_status() == wf.WF_OK
    r.close()


def _request(cfg, geom, seed, qk_raw_scale, v_raw_scale, scales, err, kernel=wf.WF_ATTN_TC):
    r = make_round(cfg, geom, wf.WF_FP8, fp8_scales=scales)
    raw, traw = raw_fn(seed, geom, torch.bfloat16, qk_raw_scale, v_raw_scale)
    out = r.new_out()
    worst = (0.0, 0.0, 0.0)
    for k in range(sch.n_rounds(cfg)):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
        out.zero_()
        r.attention(0, out, kernel)
        torch.cuda.synchronize()
        ref = round_attention(cfg, geom, k, 0, raw, qk_dtype=Fp8(*scales))
        for t, o in zip(sch.round_tasks(cfg, k), ref):
            e = err(out[t.stage].float().cpu().numpy(), o)
            worst = tuple(max(a, b) for a, b in zip(worst, e))
    assert r.sync_status() == wf.WF_OK
    r.close()
    return worst


@pytest.mark.parametrize("kernel", TC_KERNELS)
@pytest.mark.parametrize("cfg", [sch.Cfg(4, 10, 3), sch.Cfg(2, 6, -1),
                                 sch.Cfg(3, 7, 1, anchor_mode=sch.ANCHOR_ABSOLUTE)], ids=str)
def test_fp8_request_sharp_inputs(cfg, kernel):
    mx, mean, rel = _request(cfg, SMALL, 7, 2.0, 1.0, (4.0, 4.0), scaled_errors, kernel)
    assert mx <= MAX and mean <= MEAN and rel <= REL, (mx, mean, rel)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_fp8_request_bench_distribution(kernel):
    s = 1.0 / np.sqrt(128)
    mx, mean, rel = _request(sch.Cfg(4, 9, 3), SMALL, 3, s, s, (8.0, 8.0), errors, kernel)
    assert mx <= 2e-2 and mean <= 2e-3 and rel <= REL, (mx, mean, rel)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_fp8_wan_shape_sampled_rows(kernel):
    """8-bit attention at the Wan2.1-1.3B shape (S = 4, 4680-token chunks,
    12 x 128, W = 3) in a steady round with anchor re-rotation, against the
    oracle with the same e4m3 storage on sampled query rows of 3 heads.
    Absolute bars max 3.5e-3, mean 7e-4 (tests/derive_fp8_bars.py: the
    emulated e4m3 rounding of P moves these rows by max 7e-4, mean 1.5e-4;
    a planted mask mistake by max 0.0118, mean 0.0028)."""
    cfg = sch.Cfg(4, 14, 3)
    geom = Geom(3, 30, 52, 12, 128)
    heads = [0, 5, 11]
    s = 1.0 / np.sqrt(128)
    scales = (8.0, 8.0)
    r = make_round(cfg, geom, wf.WF_FP8, fp8_scales=scales)
    raw, traw = raw_fn(21, geom, torch.bfloat16, qk_scale=4 * s, v_scale=1.0, heads=heads)
    out = r.new_out()
    k_check = cfg.S + cfg.history + 2
    for k in range(k_check + 1):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
    r.attention(0, out, kernel)
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_OK
    rows = [0, 1, 127, 128, 2000, 4607, 4608, 4650, 4679]
    geom_h = Geom(3, 30, 52, len(heads), 128)
    ref = round_attention(cfg, geom_h, k_check, 0, raw, rows=rows, qk_dtype=Fp8(*scales))
    for t, o in zip(sch.round_tasks(cfg, k_check), ref):
        g = out[t.stage][rows][:, heads].float().cpu().numpy()
        mx, mean, rel = errors(g, o)
        assert mx <= 3.5e-3 and mean <= 7e-4 and rel <= REL, (t.stage, mx, mean, rel)
    r.close()
