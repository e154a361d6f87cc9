"""Derivation of the max-abs parity bars of the 8-bit attention checks
(tests/test_gpu_fp8.py, tests/test_gpu_dit.py).  Not collected by pytest;
run it by hand (a few minutes on the CPU):

    python tests/derive_fp8_bars.py

The tensor-core kernel with e4m3 pages computes what the oracle computes
with the same e4m3 storage of Q, K and V, except for one rounding the oracle
does not model: the softmax probabilities P are rounded to e4m3 before the
PV product (relative error up to 2^-4 per probability; values below the
e4m3 subnormal range vanish).  This script estimates the spread that
rounding causes by running the oracle twice -- as is, and with its dense
attention replaced by one that rounds the unnormalised probabilities
exp(s - max) to e4m3 before multiplying by V while the row sum keeps the
unrounded values, as the kernel does -- and, for the upper side, the
difference a planted mask mistake makes (every query also reading the
noisier live chunks: the reverse edges the chunk-causal mask removes).
It prints the worst (max, mean, relative L2) of |O - O_ref| / max(1, |O_ref|)
for each check.  A bar must sit above the rounding spread and at least 3x
below the mistake.  Calls only oracle/ and the seeded generators; the
probability rounding is the one step written here, from the e4m3 format
definition the oracle already uses."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import torch                                        # noqa: E402

import wf_synth                                     # noqa: E402
import oracle.dit as od                             # noqa: E402
import oracle.round as orr                          # noqa: E402
from oracle import dit                              # noqa: E402
from oracle import schedule as sch                  # noqa: E402
from oracle.attention import masked_attention       # noqa: E402
from oracle.round import Fp8, Geom, e4m3, round_attention   # noqa: E402
from gpu_helpers import errors, raw_fn, scaled_errors   # noqa: E402


def attention_p_e4m3(q, k, v, mask, scale=None):
    """Dense masked attention whose probabilities are rounded to e4m3 before
    PV (row sums from the unrounded values)."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    s = np.where(mask[None], np.matmul(q, np.swapaxes(k, -1, -2)) * scale, -np.inf)
    p = np.where(mask[None], np.exp(s - s.max(axis=-1, keepdims=True)), 0.0)
    return np.matmul(e4m3(p), v) / p.sum(axis=-1, keepdims=True)


def planted(cfg):
    return sch.Cfg(cfg.S, cfg.n_chunks, cfg.history, anchor_mode=cfg.anchor_mode,
                   use_anchor=cfg.use_anchor, mask=sch.MASK_RF)


def worst(pairs, err):
    w = [0.0, 0.0, 0.0]
    for a, b in pairs:
        w = [max(x, y) for x, y in zip(w, err(a, b))]
    return [round(x, 5) for x in w]


def attention_requests():
    geom = Geom(3, 10, 10, 2, 128)
    for cfg in (sch.Cfg(4, 10, 3), sch.Cfg(2, 6, -1), sch.Cfg(3, 7, 1, anchor_mode=sch.ANCHOR_ABSOLUTE)):
        raw, _ = raw_fn(7, geom, torch.bfloat16, 2.0, 1.0)
        fp8 = Fp8(4.0, 4.0)
        rounding, mistake = [], []
        for k in range(sch.n_rounds(cfg)):
            ref = round_attention(cfg, geom, k, 0, raw, qk_dtype=fp8)
            orr.masked_attention = attention_p_e4m3
            try:
                em = round_attention(cfg, geom, k, 0, raw, qk_dtype=fp8)
            finally:
                orr.masked_attention = masked_attention
            bad = round_attention(planted(cfg), geom, k, 0, raw, qk_dtype=fp8)
            rounding += list(zip(em, ref))
            mistake += [(b, r) for b, r, t in zip(bad, ref, sch.round_tasks(cfg, k)) if t.stage < cfg.S]
        print("attention, sharp inputs", cfg, "rounding", worst(rounding, scaled_errors),
              "mistake", worst(mistake, scaled_errors))


def wan_rows():
    cfg = sch.Cfg(4, 14, 3)
    geom = Geom(3, 30, 52, 12, 128)
    heads = [0, 5, 11]
    s = 1.0 / np.sqrt(128)
    raw, _ = raw_fn(21, geom, torch.bfloat16, qk_scale=4 * s, v_scale=1.0, heads=heads)
    geom_h = Geom(3, 30, 52, len(heads), 128)
    rows = [0, 1, 127, 128, 2000, 4607, 4608, 4650, 4679]
    k = cfg.S + cfg.history + 2
    fp8 = Fp8(8.0, 8.0)
    ref = round_attention(cfg, geom_h, k, 0, raw, rows=rows, qk_dtype=fp8)
    orr.masked_attention = attention_p_e4m3
    try:
        em = round_attention(cfg, geom_h, k, 0, raw, rows=rows, qk_dtype=fp8)
    finally:
        orr.masked_attention = masked_attention
    bad = round_attention(planted(cfg), geom_h, k, 0, raw, rows=rows, qk_dtype=fp8)
    tasks = sch.round_tasks(cfg, k)
    print("attention, Wan2.1-1.3B rows", "rounding", worst(zip(em, ref), errors),
          "mistake", worst([(b, r) for b, r, t in zip(bad, ref, tasks) if t.stage < cfg.S], errors))


def dit_requests():
    cfg = sch.Cfg(4, 6, 3)
    dims = dit.Dims(dim=256, heads=2, head_dim=128, ffn=512, layers=2, channels=16, freq=256)
    grid = (3, 8, 10)
    for seed, linear_fp8, kv in ((13, False, (4.0, 4.0)), (15, True, None), (15, True, (4.0, 4.0))):
        params = wf_synth.dit_params(seed, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                     std=0.02)

        def lat(c, s):
            return wf_synth.latent(seed, c, s, 16, 3, 16, 20).double().numpy()

        def run(mask_fn, c=cfg):
            m = dit.Model(c, grid, dims, dit.weights_from(params), [1000.0, 750.0, 500.0, 250.0],
                          bf16_points=True, kv_fp8=kv, linear_fp8=linear_fp8)
            od.masked_attention = mask_fn
            try:
                outs = []
                for k in range(sch.n_rounds(c)):
                    x0, em = m.round(k, lat(k, -1), [lat(k - s, s) for s in range(4)])
                    outs += x0 + ([em] if em is not None else [])
            finally:
                od.masked_attention = masked_attention
            return outs

        ref = run(masked_attention)
        em = run(attention_p_e4m3) if kv else ref
        bad = run(lambda q, k, v, mask: masked_attention(q, k, v, np.ones_like(mask)))
        print("DiT request", "e4m3 linears" if linear_fp8 else "bf16 linears",
              "e4m3 attention" if kv else "bf16 attention",
              "rounding", worst(zip(em, ref), scaled_errors), "mistake", worst(zip(bad, ref), scaled_errors))


if __name__ == "__main__":
    attention_requests()
    wan_rows()
    dit_requests()
