"""Shared helpers of the GPU parity tests: drive the C ABI through a request
with seeded inputs and compare against the oracle."""

import numpy as np
import torch

import chunk_causal_dit_round_b300 as wf
import wf_synth
from oracle import schedule as sch
from oracle.round import Geom


def make_round(cfg: sch.Cfg, geom: Geom, dtype, layers=1, fp8_scales=(1.0, 1.0)):
    return wf.Round(cfg.S, geom.chunk_tokens, geom.heads, geom.head_dim, cfg.history, fp8_scales=fp8_scales,
                    n_chunks=cfg.n_chunks, layers=layers, grid=geom.grid, dtype=dtype,
                    use_anchor=cfg.use_anchor, anchor_mode=cfg.anchor_mode,
                    rope_theta=geom.theta, mask=cfg.mask, store_extra=cfg.store_extra,
                    rope_split=geom.rope_split,
                    schedule=wf.WF_SCHED_SEQUENTIAL if cfg.sequential else wf.WF_SCHED_WAVEFRONT)


def raw_fn(seed, geom: Geom, tdtype, qk_scale=1.0, v_scale=1.0, heads=None):
    """raw(chunk, stage, layer) -> fp64 numpy [N_C, 3, H', D] of exactly the
    values the GPU reads (rounded to the storage dtype first)."""
    cache = {}

    def torch_raw(chunk, stage, layer):
        key = (chunk, stage, layer)
        if key not in cache:
            x = wf_synth.qkv_raw(seed, chunk, stage, layer, geom.chunk_tokens, geom.heads,
                                 geom.head_dim)
            x[:, 0:2] *= qk_scale
            x[:, 2] *= v_scale
            cache[key] = x.to(tdtype)
        return cache[key]

    def raw(chunk, stage, layer):
        x = torch_raw(chunk, stage, layer).double().numpy()
        return x if heads is None else x[:, :, heads]

    return raw, torch_raw


def fill_qkv(r: wf.Round, info, torch_raw, layer, qkv=None):
    if qkv is None:
        qkv = r.new_qkv()
    for i in range(info.n_tasks):
        c, s = info.task_chunk[i], info.task_stage[i]
        qkv[s].copy_(torch_raw(c, s, layer))
    return qkv


def errors(gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(gpu.astype(np.float64) - ref)
    rel = np.linalg.norm(gpu.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-30)
    return float(d.max()), float(d.mean()), float(rel)


def scaled_errors(gpu: np.ndarray, ref: np.ndarray):
    """Errors of O / max(1, |O|): the stated absolute tolerance for outputs of
    magnitude <= 1, relative beyond.  An absolute 2e-2 cannot hold for large
    outputs: rounding O to bf16 errs by up to half an ulp (2^-6 ~ 0.0156 for
    |O| in [4, 8)), and rounding P to bf16 before PV moves O by up to
    2^-9 max|v| more (another 0.0156 when |v| reaches 8), so the two together
    pass 2e-2 once |O| >= 4."""
    g = gpu.astype(np.float64)
    d = np.abs(g - ref) / np.maximum(1.0, np.abs(ref))
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    return float(d.max()), float(d.mean()), float(rel)
