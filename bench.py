#!/usr/bin/env python3
"""Benchmark of one wavefront round of chunk-wise causal attention on B300.

Workload (default ``wan13_attn``): the Wan2.1-1.3B attention layer of
"Wave Forcing" (S = 4 denoising stages + store = 5 tasks per round; chunks of
3 latent frames x 30 x 52 patches = 4680 tokens; 12 heads x 128; bf16 Q/K/V
~ N(0,1)/sqrt(128) with 3D RoPE; history window of 3 chunks plus the anchor),
in steady-state rounds of a 133-chunk request (the paper's 399-latent-frame
video).  One step = one round: wf_round_step (host schedule + page ring),
wf_qkv_rope_publish (RoPE + paged K/V placement + anchor re-rotation) and
wf_round_attention (one launch over all 5 tasks).  Inputs are seeded
synthetic tensors already resident in HBM; each step reads > 126 MB (larger
than L2), so no explicit flush is needed.

Prints one JSON line (rank 0): the attention TFLOP/s with the attention
kernel's roofline (CUDA-event time per launch against the measured peak),
the publish kernel's GB/s against the measured HBM bandwidth, the same
metric end to end with host buffers (``e2e``), the clocks seen during the
timed region, the oracle timed on the host cores (``cpu_baseline``),
batched requests (``streams``: the attention layer; ``dit_streams``: whole
DiT rounds), and the whole DiT round (chunks/s, frames/s) for the bf16 model
(``dit``), the 8-bit one (``dit_w8a8``), the 5-step long rollout
(``dit_s5``) and the 14B-scale QKV + attention stack (``qkv_attn14b``).
``--config`` selects single workloads;
``--impl reference`` times the CPU oracle on a bounded sample of the same
round instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunk-causal attention TFLOP/s (% bf16 peak); DiT chunks/s per 1F1C round"
UNIT = "TFLOP/s"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one steady
# attn_tc_kernel launch of the wan13_attn round (bf16 and e4m3 pages), from an
# ncu capture, with the sha256 (first 16 hex digits) of the kernel's sources
# at capture time.  The bench reports the figure only while the sources still
# hash to that value, so a changed kernel reports null until it is captured
# again.
ATTN_TC_SOURCES = ("chunk_causal_dit_round_b300/csrc/attn_tc.cu",
                   "chunk_causal_dit_round_b300/csrc/wf_ptx.cuh")
ATTN_TC_TRAFFIC = {"bf16": (5.2925e8, "d47bd0f5fe615e78"), "e4m3": (2.1823e8, "d47bd0f5fe615e78")}


# Video frames of a request: "Wave Forcing", App. C (VBench-Long protocol),
# saves 1593 video frames for 399 latent frames -- the first latent frame
# decodes to one video frame and every later one to four -- so a chunk of
# grid_t latent frames adds 4 grid_t video frames in steady state.
def video_frames(n_chunks, latent_frames_per_chunk=3):
    return 1 + (n_chunks * latent_frames_per_chunk - 1) * 4


def frames_per_s(chunks_per_s, latent_frames_per_chunk=3):
    return 4 * latent_frames_per_chunk * chunks_per_s


def eta_slot(n_chunks, S, sequential=False):
    """Useful fraction of a request's stage slots ("Wave Forcing", App. B.4
    Eq. 16): a wavefront request of N chunks takes N + S rounds of S + 1
    slots for N (S + 1) tasks; the sequential schedule keeps one of S + 1
    stage replicas busy."""
    return 1 / (S + 1) if sequential else n_chunks / (n_chunks + S)


def _p90(xs):
    """90th percentile (nearest rank) of a list of times."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, math.ceil(0.9 * len(ys)) - 1))]


def _sources_sha16(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def attn_traffic(kind):
    """(bytes, note): the captured DRAM traffic of one launch, or None when
    the kernel's sources changed since the capture."""
    nbytes, sha = ATTN_TC_TRAFFIC[kind]
    now = _sources_sha16(ATTN_TC_SOURCES)
    if now != sha:
        return None, f"kernel sources {now} differ from the captured {sha}: not re-captured yet"
    return nbytes, f"ncu capture of one steady launch, kernel sources {sha}"

CONFIGS = {
    # name: (S, grid (t,h,w), heads, head_dim, history W)
    "wan13_attn": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3,
                       desc="Wan2.1-1.3B attention layer, S=4 (5 tasks/round), 4680-token chunks, "
                            "12x128 heads, W=3 + anchor, bf16"),
    "wan13_attn_fp8": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, fp8=(8.0, 8.0),
                           desc="the same round with 8-bit attention: Q and K/V pages in e4m3 "
                                "(x8 scales), P in e4m3, bf16 Q/K/V input and output"),
}


DIT_CONFIGS = {
    # name: Wan2.1-shaped DiT rounds (random-init weights ~ N(0, 0.02), bf16)
    "dit13": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                  layers=30, n_chunks=64, steps=[1000.0, 750.0, 500.0, 250.0],
                  desc="random-init Wan2.1-1.3B-shaped DiT, 4-step (S=4), 30 blocks, dim 1536, "
                       "12x128 heads, FFN 8960, 4680-token chunks, W=3 + anchor, 64 chunks"),
    "dit13_s5": dict(S=5, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                     layers=30, n_chunks=135, steps=[1000.0, 800.0, 600.0, 400.0, 200.0],
                     desc="long rollout, 5-step (S=5), same 1.3B shapes, 135 chunks, paged K/V "
                          "ring with oldest-chunk eviction, W=3 + anchor"),
    "dit13_fp8": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                      layers=30, n_chunks=64, steps=[1000.0, 750.0, 500.0, 250.0], fp8=(4.0, 4.0),
                      desc="as dit13 with 8-bit attention: e4m3 Q and K/V pages (x4 scales), "
                           "e4m3 P; linear layers bf16"),
    "dit13_w8a8": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                       layers=30, n_chunks=64, steps=[1000.0, 750.0, 500.0, 250.0], fp8=(4.0, 4.0),
                       linear_fp8=True,
                       desc="as dit13 with 8-bit attention and 8-bit linear layers (e4m3 weights "
                            "per output channel, e4m3 activations); patch embedding and head bf16"),
    # comparison graphs on the same model and kernels
    "dit13_rf": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                     layers=30, n_chunks=64, steps=[1000.0, 750.0, 500.0, 250.0], mask=1,
                     desc="as dit13 with Rolling Forcing's full active-window mask (reverse "
                          "edges to noisier live chunks), one round per chunk"),
    "dit13_seq": dict(S=4, grid=(3, 30, 52), heads=12, head_dim=128, history=3, dim=1536, ffn=8960,
                      layers=30, n_chunks=64, steps=[1000.0, 750.0, 500.0, 250.0], sequential=True,
                      desc="as dit13 run sequentially (NF1C): each chunk's 4 denoising forwards "
                           "and its store pass, one task per forward"),
}


QKV_ATTN_CONFIGS = {
    "qkv_attn14b": dict(S=4, grid=(3, 30, 52), heads=40, head_dim=128, history=3, dim=5120,
                        layers=40, n_chunks=64,
                        desc="14B-scale QKV + attention stack: dim 5120, 40 heads x 128, S=4, "
                             "4680-token chunks, W=3 + anchor, 40 layers, random-init bf16 "
                             "weights ~ N(0, 0.02)"),
}


def run_qkv_attn(args, name, rank, world, steps=None, warmup=None):
    """Steady rounds of the per-layer P and attention of a 14B-scale model:
    for each layer, wf_qkv_proj_rope_publish (QKV GEMM 5120 -> 15360, the
    q/k RMSNorm, RoPE + paged publish) and wf_round_attention; the normalised
    layer input is a synthetic N(0, 1) bf16 activation (the rest of the block
    is out of this workload)."""
    import torch
    import chunk_causal_dit_round_b300 as wf

    cfg = QKV_ATTN_CONFIGS[name]
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    S, W = cfg["S"], cfg["history"]
    L = getattr(args, "layers", None) or cfg["layers"]
    NC = math.prod(cfg["grid"])
    H, D, dim = cfg["heads"], cfg["head_dim"], cfg["dim"]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    k_steady = S + W + 2
    n_chunks = max(cfg["n_chunks"], k_steady + warmup + steps + 1)
    r = wf.Round(S, NC, H, D, W, n_chunks=n_chunks, layers=L, grid=cfg["grid"], dtype=wf.WF_BF16)
    g = torch.Generator(device=dev)
    g.manual_seed(777 + rank)
    ws = [(torch.randn((3 * dim, dim), generator=g, device=dev) * 0.02).to(torch.bfloat16)
          for _ in range(L)]
    bs = [(torch.randn((3 * dim,), generator=g, device=dev) * 0.02).to(torch.bfloat16)
          for _ in range(L)]
    # q / k RMSNorm gains of the standard Wan2.1 block: 1 + N(0, 0.02^2)
    nqs = [(1 + torch.randn((dim,), generator=g, device=dev) * 0.02).to(torch.bfloat16)
           for _ in range(L)]
    nks = [(1 + torch.randn((dim,), generator=g, device=dev) * 0.02).to(torch.bfloat16)
           for _ in range(L)]
    xs = [torch.randn((S + 1, NC, dim), generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
    out = torch.empty((S + 1, NC, dim), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def one_round(i):
        info = r.step()
        for l in range(L):
            r.publish_proj(l, xs[i % 2], ws[l], bs[l], nqs[l], nks[l], stream)
            r.attention(l, out, wf.WF_ATTN_TC, stream)
        return info

    for i in range(k_steady + warmup):
        one_round(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    flops = 0.0
    launches = 0
    prev_anchor = r.info.anchor_tpos
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        for j in range(steps):
            evs[j][0].record(stream)
            info = one_round(j)
            evs[j][1].record(stream)
            T = info.n_tasks * NC
            flops += L * (info.attn_flops + 2.0 * T * dim * 3 * dim)
            # per layer: QKV GEMM, q/k RMSNorm + RoPE + publish, attention, and
            # the anchor re-rotation in rounds where the window moved
            moved = info.anchor_tpos >= 0 and info.anchor_tpos != prev_anchor
            launches += (4 if moved else 3) * L
            prev_anchor = info.anchor_tpos
        torch.cuda.synchronize()
    st = r.sync_status()
    if st != wf.WF_OK:
        raise RuntimeError(f"device status {st}")
    per = [a.elapsed_time(b) for a, b in evs]
    ms, = max_over_ranks([sum(per)], world, dev)
    peak, src = _sustained_peak()
    tf = flops / (ms * 1e-3) / 1e12
    res = {"workload": name, "desc": cfg["desc"], "layers": L,
           "value": round(world * steps / (ms * 1e-3), 3), "unit": "chunks/s",
           "value_p50": round(world * 1e3 / statistics.median(per), 3),
           "round_ms_p50": round(statistics.median(per), 3), "round_ms_p90": round(_p90(per), 3),
           "rounds": steps,
           "flops_per_round": flops / steps,
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                        "peak_source": f"{src} bf16 dense (sustained)"},
           "gpu_launches": launches, "clocks": clk.summary()}
    del r, ws, xs
    torch.cuda.empty_cache()
    return res


STREAM_SHAPES = {
    # chunk geometries of the batched-requests measurement: the Wan2.1-1.3B
    # chunk (3 latent frames) and a one-latent-frame chunk
    "chunk4680": dict(grid=(3, 30, 52), desc="3 latent frames x 30 x 52 patches"),
    "chunk1560": dict(grid=(1, 30, 52), desc="1 latent frame x 30 x 52 patches"),
    # a quarter-size frame (240 x 416 video): one request's round has 120
    # work units, fewer than the SMs
    "chunk390": dict(grid=(1, 15, 26), desc="1 latent frame x 15 x 26 patches"),
}


def run_streams(args, rank, world, counts=(1, 2, 4, 8), steps=10, warmup=3):
    """Several requests batched into one round (wf_group_*): for R requests
    of the Wan2.1-1.3B attention layer (S = 4, 12 x 128 heads, W = 3 +
    anchor), each steady round runs one batched publication (RoPE + paged
    placement of all R (S+1) tasks) and one batched attention launch; every
    request completes one chunk per round, so chunks/s = R / round time.
    Measured at two chunk sizes; the gain over R = 1 is the occupancy the
    batching recovers."""
    import torch
    import chunk_causal_dit_round_b300 as wf

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    base = CONFIGS["wan13_attn"]
    S, W, H, D = base["S"], base["history"], base["heads"], base["head_dim"]
    k_steady = S + W + 2
    stream = torch.cuda.current_stream()
    out = {}
    for name, shp in STREAM_SHAPES.items():
        NC = math.prod(shp["grid"])
        rows = []
        for R in counts:
            grp = wf.Group(R, S, NC, H, D, W, n_chunks=k_steady + warmup + 400, grid=shp["grid"],
                           dtype=wf.WF_BF16, device=dev)
            g = torch.Generator(device=dev)
            g.manual_seed(99 + R)
            qkvs = []
            for _ in range(2):
                x = torch.randn((R, S + 1, NC, 3, H, D), generator=g, device=dev)
                qkvs.append((x / math.sqrt(D)).to(torch.bfloat16))
                del x
            o = grp.new_out()
            mask = (1 << R) - 1

            def one(i):
                fl = 0.0
                for r in grp.rounds:
                    fl += r.step().attn_flops
                grp.publish(mask, 0, qkvs[i % 2], stream)
                grp.attention(mask, 0, o, wf.WF_ATTN_TC, stream)
                return fl

            for i in range(k_steady + warmup):
                one(i)
            torch.cuda.synchronize()
            # time at least ~0.3 s per row so the clock sampler sees it
            t0 = time.perf_counter()
            one(0)
            torch.cuda.synchronize()
            n_t = max(steps, int(0.3 / max(time.perf_counter() - t0, 1e-4)))
            n_t = min(n_t, grp.rounds[0].n_left())
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_t)]
            flops = 0.0
            with ClockSampler(dev.index) as clk:
                torch.cuda.synchronize()
                for j in range(n_t):
                    evs[j][0].record(stream)
                    flops += one(j)
                    evs[j][1].record(stream)
                torch.cuda.synchronize()
            st = grp.rounds[0].sync_status()
            if st != wf.WF_OK:
                raise RuntimeError(f"device status {st}")
            per = [a.elapsed_time(b) for a, b in evs]
            ms, = max_over_ranks([sum(per)], world, dev)
            rows.append({"requests": R, "chunks_per_s": round(world * R * n_t / (ms * 1e-3), 2),
                         "round_ms": round(ms / n_t, 4), "rounds": n_t,
                         "attn_tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                         "clocks": clk.summary()})
            grp.close()
            del grp, qkvs, o
            torch.cuda.empty_cache()
        base1 = rows[0]["chunks_per_s"]
        for r_ in rows:
            r_["vs_one_request"] = round(r_["chunks_per_s"] / base1, 3)
        out[name] = {"chunk_tokens": NC, "desc": shp["desc"], "rows": rows}
    return {"workload": "batched requests, Wan2.1-1.3B attention layer (publish + attention per round)",
            "unit": "chunks/s", "shapes": out, "gpu_launches_per_round": 2}


def measure_peaks(n=8192, seconds=4.0):
    """The dense GEMM peaks of this GPU for the 8-bit rooflines, measured as
    the bf16 denominator is: a library GEMM (cuBLASLt through torch) at
    n^3, the best of 10 launches (burst) and back-to-back launches for
    ``seconds`` (sustained), for e4m3 (torch._scaled_mm, unit scales, bf16
    out) and bf16.  A denominator measurement, not a workload of this
    library."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    one = torch.ones((), device=dev)
    a8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    ab = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    bb = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    fns = {"e4m3": lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one,
                                            out_dtype=torch.bfloat16),
           "bf16": lambda: ab @ bb}
    res = {}
    for name, fn in fns.items():
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        res[name] = {"burst_tflops": round(2 * n ** 3 / (best * 1e-3) / 1e12, 1)}
        if seconds <= 0:          # burst launches only (e.g. for a short profiler capture)
            continue
        with ClockSampler(dev.index) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0, count = time.time(), 0
            e0.record()
            while time.time() - t0 < seconds:
                for _ in range(20):
                    fn()
                count += 20
                torch.cuda.synchronize()
            e1.record()
            torch.cuda.synchronize()
        res[name].update({"sustained_tflops": round(2 * n ** 3 * count / (e0.elapsed_time(e1) * 1e-3) / 1e12, 1),
                          "clocks_sustained": clk.summary()})
    return {"workload": f"library dense GEMM {n}^3 (cuBLASLt through torch)", "peaks": res}


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of per-rank timings over all replicas (one
    process per GPU, independent replicas; the slowest rank sets the
    whole-job time).  With world == 1 the values come back unchanged."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def _sustained_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return d["bf16_tflops_sustained"], "measured"
    return 1400.0, "fallback"


def _dit_params(g, dev, dim, ffn, L, C):
    """Random-init Wan2.1-shaped DiT weights, bf16 ~ N(0, 0.02); q / k
    RMSNorm gains 1 + N(0, 0.02^2)."""
    import torch

    def rnd(*shape, std=0.02):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    P = {"patch_w": rnd(dim, 4 * C), "patch_b": rnd(dim), "t1_w": rnd(dim, 256), "t1_b": rnd(dim),
         "t2_w": rnd(dim, dim), "t2_b": rnd(dim), "tp_w": rnd(6 * dim, dim), "tp_b": rnd(6 * dim),
         "head_w": rnd(4 * C, dim), "head_b": rnd(4 * C), "head_mod": rnd(2, dim)}
    for k_, shp in (("qkv_w", (3 * dim, dim)), ("qkv_b", (3 * dim,)), ("o_w", (dim, dim)),
                    ("o_b", (dim,)), ("f1_w", (ffn, dim)), ("f1_b", (ffn,)), ("f2_w", (dim, ffn)),
                    ("f2_b", (dim,)), ("mod", (6, dim))):
        P[k_] = [rnd(*shp) for _ in range(L)]
    for k_ in ("nq", "nk"):
        P[k_] = [(1 + rnd(dim).float()).to(torch.bfloat16) for _ in range(L)]
    return P


def run_dit_streams(args, rank, world, counts=(1, 2, 4, 8), steps=10, warmup=3):
    """Several requests batched into whole DiT rounds (wf_group_dit_round):
    R requests of the random-init Wan2.1-1.3B-shaped DiT (dit13's model, S = 4,
    30 blocks), each steady round one group DiT pass over all R (S+1) tasks;
    every request completes one chunk per round, so chunks/s = R / round time.
    At small chunks one request's GEMMs and attention fill a fraction of the
    SMs; batching recovers it."""
    import torch
    import chunk_causal_dit_round_b300 as wf

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = DIT_CONFIGS["dit13"]
    S, W, H, D, dim, ffn = cfg["S"], cfg["history"], cfg["heads"], cfg["head_dim"], cfg["dim"], cfg["ffn"]
    L = getattr(args, "layers", None) or cfg["layers"]
    C = 16
    k_steady = S + W + 2
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + rank)
    P = _dit_params(g, dev, dim, ffn, L, C)
    out = {}
    for name in ("chunk390", "chunk1560"):
        shp = STREAM_SHAPES[name]
        NC = math.prod(shp["grid"])
        latent = C * shp["grid"][0] * 4 * shp["grid"][1] * shp["grid"][2]
        rows = []
        for R in counts:
            grp = wf.Group(R, S, NC, H, D, W, n_chunks=k_steady + warmup + 400, layers=L,
                           grid=shp["grid"], dtype=wf.WF_BF16, device=dev)
            model = wf.GroupDit(grp, P, ffn=ffn, channels=C, freq=256, timesteps=cfg["steps"])
            z = torch.randn((R, latent), generator=g, device=dev)
            eps = torch.randn((R, S, latent), generator=g, device=dev)
            chunk = torch.empty((R, latent), device=dev)
            mask = (1 << R) - 1

            def one():
                for r in grp.rounds:
                    r.step()
                model.round(mask, z, eps, None, chunk, stream)

            for _ in range(k_steady + warmup):
                one()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            one()
            torch.cuda.synchronize()
            n_t = max(steps, int(0.3 / max(time.perf_counter() - t0, 1e-4)))
            n_t = min(n_t, grp.rounds[0].n_left())
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with ClockSampler(dev.index) as clk:
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(n_t):
                    one()
                e1.record(stream)
                torch.cuda.synchronize()
            st = grp.rounds[0].sync_status()
            if st != wf.WF_OK:
                raise RuntimeError(f"device status {st}")
            ms, = max_over_ranks([e0.elapsed_time(e1)], world, dev)
            rows.append({"requests": R, "chunks_per_s": round(world * R * n_t / (ms * 1e-3), 2),
                         "round_ms": round(ms / n_t, 3), "rounds": n_t, "clocks": clk.summary()})
            del model
            grp.close()
            del grp, z, eps, chunk
            torch.cuda.empty_cache()
        base1 = rows[0]["chunks_per_s"]
        for r_ in rows:
            r_["vs_one_request"] = round(r_["chunks_per_s"] / base1, 3)
        out[name] = {"chunk_tokens": NC, "desc": shp["desc"], "rows": rows}
    return {"workload": f"batched requests, whole DiT rounds ({cfg['desc']}; chunk size as listed)",
            "layers": L, "unit": "chunks/s", "shapes": out,
            "gpu_launches_per_round": 4 + 8 * L}


def run_dit(args, name, rank, world, steps=None, warmup=None):
    """Steady wavefront rounds of the whole DiT forward (wf_dit_round): per
    layer LN + modulation, QKV projection + RoPE + paged publish, round
    attention, output projection + gated residual, LN, FFN; then the head and
    the stage transition.  One completed chunk per steady round (1F1C)."""
    import torch
    import chunk_causal_dit_round_b300 as wf

    cfg = DIT_CONFIGS[name]
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    S, W = cfg["S"], cfg["history"]
    L = getattr(args, "layers", None) or cfg["layers"]
    NC = math.prod(cfg["grid"])
    H, D, dim, ffn = cfg["heads"], cfg["head_dim"], cfg["dim"], cfg["ffn"]
    C = 16
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    seq = cfg.get("sequential", False)
    per_step = S + 1 if seq else 1          # rounds (forward passes) per completed chunk
    k_steady = (W + 2) * (S + 1) if seq else S + W + 2
    n_chunks = max(cfg["n_chunks"], (k_steady // per_step) + warmup + steps + 4)
    r = wf.Round(S, NC, H, D, W, n_chunks=n_chunks, layers=L, grid=cfg["grid"],
                 dtype=wf.WF_FP8 if cfg.get("fp8") else wf.WF_BF16,
                 fp8_scales=cfg.get("fp8") or (1.0, 1.0), mask=cfg.get("mask", 0),
                 schedule=wf.WF_SCHED_SEQUENTIAL if seq else wf.WF_SCHED_WAVEFRONT)
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + rank)
    P = _dit_params(g, dev, dim, ffn, L, C)
    model = wf.Dit(r, P, ffn=ffn, channels=C, freq=256, timesteps=cfg["steps"],
                   linear_fp8=cfg.get("linear_fp8", False))
    latent = C * cfg["grid"][0] * 4 * cfg["grid"][1] * cfg["grid"][2]
    n_in = 3
    zs = [torch.randn(latent, generator=g, device=dev) for _ in range(n_in)]
    epss = [torch.randn((S, latent), generator=g, device=dev) for _ in range(n_in)]
    chunk = torch.empty(latent, device=dev)
    stream = torch.cuda.current_stream()

    attn_total = [0.0]

    def round_flops(info):
        T = info.n_tasks * NC
        lin = 2.0 * T * (3 * dim * dim + dim * dim + 2 * dim * ffn) * L
        attn_total[0] += info.attn_flops * L
        return info.attn_flops * L + lin + 2.0 * T * (4 * C) * dim * 2

    i = 0
    for _ in range(k_steady + warmup * per_step):
        r.step()
        model.round(zs[i % n_in], epss[i % n_in], None, chunk, stream)
        i += 1
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    flops = 0.0
    launches = 0
    prev_anchor = r.info.anchor_tpos
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        t0.record(stream)
        for j in range(steps):
            evs[j][0].record(stream)
            for _ in range(per_step):
                info = r.step()
                model.round(zs[i % n_in], epss[i % n_in], None, chunk, stream)
                flops += round_flops(info)
                # patchify, patch GEMM, head LN, head GEMM; 8 per layer (LN,
                # QKV GEMM, q/k RMSNorm, attention, output GEMM, LN, FFN1,
                # FFN2); plus a re-rotation launch per layer when the anchor moved
                moved = info.anchor_tpos >= 0 and info.anchor_tpos != prev_anchor
                launches += 4 + 8 * L + (L if moved else 0)
                prev_anchor = info.anchor_tpos
                i += 1
            evs[j][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    st = r.sync_status()
    if st != wf.WF_OK:
        raise RuntimeError(f"device status {st}")
    per = sorted(a.elapsed_time(b) for a, b in evs)

    # end to end through the public API with host buffers: each chunk's fresh
    # noise and transition draws go up from pinned memory, the finished clean
    # chunk comes back
    h_z = torch.empty(latent, dtype=torch.float32).pin_memory()
    h_eps = torch.empty((S, latent), dtype=torch.float32).pin_memory()
    h_z.copy_(zs[0].cpu())
    h_eps.copy_(epss[0].cpu())
    h_out = torch.empty(latent, dtype=torch.float32).pin_memory()
    d_z, d_eps = torch.empty_like(zs[0]), torch.empty_like(epss[0])
    e2e_steps = steps                       # as many chunks as the device-timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk_e2e:
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(e2e_steps):
            for _ in range(per_step):
                d_z.copy_(h_z, non_blocking=True)
                d_eps.copy_(h_eps, non_blocking=True)
                r.step()
                model.round(d_z, d_eps, None, chunk, stream)
            h_out.copy_(chunk, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
    ms, e2e_ms = max_over_ranks([t0.elapsed_time(t1), e0.elapsed_time(e1)], world, dev)
    chunks_s = world * steps / (ms * 1e-3)
    peak, src = _sustained_peak()
    peak_kind = "bf16 dense (sustained)"
    if cfg.get("fp8"):
        # attention (and with e4m3 linears the linear layers) run on the e4m3
        # pipe, 2 x bf16 nominal: the bound is the time each part would take
        # at its own peak
        fa = attn_total[0]                       # attention FLOPs of the timed rounds
        lin_x = 2.0 if cfg.get("linear_fp8") else 1.0
        t_min = fa / (2 * peak) + (flops - fa) / (lin_x * peak)
        peak_kind = (f"attention at 2 x and linears at {lin_x:g} x measured bf16 (sustained)")
        peak = flops / t_min
    tf = flops / steps / (statistics.median(per) * 1e-3) / 1e12
    res = {"workload": name, "desc": cfg["desc"], "layers": L, "value": round(chunks_s, 3),
           "unit": "chunks/s", "value_stat": "timed chunks / whole timed region",
           "value_p50": round(world * 1e3 / statistics.median(per), 3),
           "forwards_per_chunk_timed": per_step,
           "e2e": {"value": round(world * e2e_steps / (e2e_ms * 1e-3), 3), "unit": "chunks/s",
                   "h2d_bytes_per_step": per_step * (h_z.numel() + h_eps.numel()) * 4,
                   "d2h_bytes_per_step": h_out.numel() * 4, "steps": e2e_steps,
                   "clocks": clk_e2e.summary()},
           "frames_per_s": round(frames_per_s(chunks_s, cfg["grid"][0]), 2),
           "ms_per_chunk_p50": round(statistics.median(per), 3),
           "ms_per_chunk_p90": round(_p90(per), 3),
           "chunks_timed": steps,
           "eta_slot": round(eta_slot(cfg["n_chunks"], S, seq), 4),
           "flops_per_round": flops / steps,
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": round(peak, 1),
                        "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                        "peak_source": f"{src} {peak_kind}"},
           "gpu_launches": launches, "clocks": clk.summary()}
    del model, r, P
    torch.cuda.empty_cache()
    return res


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1800.0), d.get("hbm_gbs", 6400.0), "measured"
    return 1800.0, 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.out = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self.out = open(self.path, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        if self.out is not None:
            self.out.close()
            self.out = None

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def steady_plan(wf, cfg, n_chunks):
    fp8 = cfg.get("fp8")
    return wf.Round(cfg["S"], math.prod(cfg["grid"]), cfg["heads"], cfg["head_dim"], cfg["history"],
                    n_chunks=n_chunks, layers=1, grid=cfg["grid"],
                    dtype=wf.WF_FP8 if fp8 else wf.WF_BF16, fp8_scales=fp8 or (1.0, 1.0))


def run_ours(args, rank, world):
    import torch
    import chunk_causal_dit_round_b300 as wf

    cfg = CONFIGS[args.config]
    S, W = cfg["S"], cfg["history"]
    NC = math.prod(cfg["grid"])
    H, D = cfg["heads"], cfg["head_dim"]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    k_steady = S + W + 2                      # anchor present, window shifting, all tasks live
    e2e_steps = args.e2e_steps
    n_chunks = max(133, k_steady + args.warmup + args.steps + e2e_steps + 2)
    r = steady_plan(wf, cfg, n_chunks)
    stream = torch.cuda.current_stream()

    # seeded synthetic inputs, resident in HBM: a ring of distinct rounds
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    n_in = 3
    qkvs = []
    for _ in range(n_in):
        x = torch.randn((S + 1, NC, 3, H, D), generator=g, device=dev, dtype=torch.float32)
        qkvs.append((x / math.sqrt(D)).to(torch.bfloat16))
        del x
    out = r.new_out()

    kernel = {"auto": wf.WF_ATTN_AUTO, "tc": wf.WF_ATTN_TC,
              "simt": wf.WF_ATTN_SIMT}[getattr(args, "attn_kernel", "auto")]

    def step(i, qkv=None):
        info = r.step()
        if info is None:
            raise RuntimeError("request exhausted")
        r.publish(0, qkv if qkv is not None else qkvs[i % n_in], stream)
        r.attention(0, out, kernel, stream)
        return info

    # fill the pipeline (untimed): rounds 0 .. k_steady-1
    for i in range(k_steady):
        step(i)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    # ---- timed: device-resident inputs -----------------------------------
    ev_attn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    ev_pub = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    flops = 0.0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(args.steps):
            info = r.step()
            ev_pub[i].record(stream)
            r.publish(0, qkvs[i % n_in], stream)
            ev_attn[i][0].record(stream)
            r.attention(0, out, kernel, stream)
            ev_attn[i][1].record(stream)
            flops += info.attn_flops
        t1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    ms = t0.elapsed_time(t1)
    attn_ms = [a.elapsed_time(b) for a, b in ev_attn]
    pub_ms = [a.elapsed_time(b[0]) for a, b in zip(ev_pub, ev_attn)]
    st = r.sync_status()
    if st != wf.WF_OK:
        raise RuntimeError(f"device status {st}")

    # ---- timed: end to end through the C ABI with host buffers ------------
    # Every round's Q/K/V go up from pinned host memory and its output comes
    # back.  Two device buffers each way; each upload is split over two copy
    # streams (one copy engine alone does not fill the host link) and a third
    # stream reads the outputs back: round i+1's upload and round i-1's
    # readback overlap round i's kernels.
    host_in = torch.empty_like(qkvs[0], device="cpu").pin_memory()
    host_in.copy_(qkvs[0].cpu())
    host_out = [torch.empty(out.shape, dtype=out.dtype, device="cpu").pin_memory() for _ in range(2)]
    dev_in = [torch.empty_like(qkvs[0]) for _ in range(2)]
    dev_out = [r.new_out() for _ in range(2)]
    ups, down = [torch.cuda.Stream(), torch.cuda.Stream()], torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done = [[ev(), ev()], [ev(), ev()]]        # [buffer][copy stream]
    comp_done, d2h_done = [ev(), ev()], [ev(), ev()]
    flat_in = host_in.view(-1)
    half = flat_in.numel() // 2

    def upload(nb):
        for u, (lo, hi) in enumerate(((0, half), (half, flat_in.numel()))):
            with torch.cuda.stream(ups[u]):
                dev_in[nb].view(-1)[lo:hi].copy_(flat_in[lo:hi], non_blocking=True)
                h2d_done[nb][u].record(ups[u])

    # the host link's rate for one copy of this size, one and two streams
    link = {}
    for n_str in (1, 2):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        l0.record(stream)
        for u in range(n_str):
            ups[u].wait_stream(stream)
        if n_str == 1:
            with torch.cuda.stream(ups[0]):
                dev_in[0].copy_(host_in, non_blocking=True)
        else:
            upload(0)
        for u in range(n_str):
            stream.wait_stream(ups[u])
        l1.record(stream)
        torch.cuda.synchronize()
        link[n_str] = host_in.numel() * host_in.element_size() / (l0.elapsed_time(l1) * 1e-3) / 1e9
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_flops = 0.0
    torch.cuda.synchronize()
    e0.record(stream)
    for u in ups:
        u.wait_stream(stream)
    down.wait_stream(stream)
    upload(0)
    for i in range(e2e_steps):
        b = i % 2
        if i + 1 < e2e_steps:
            nb = (i + 1) % 2
            if i >= 1:
                for u in ups:
                    u.wait_event(comp_done[nb])          # round i-1 has read dev_in[nb]
            upload(nb)
        for u in range(2):
            stream.wait_event(h2d_done[b][u])
        if i >= 2:
            stream.wait_event(d2h_done[b])                # round i-2's output is home
        info = r.step()
        r.publish(0, dev_in[b], stream)
        r.attention(0, dev_out[b], kernel, stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(comp_done[b])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            d2h_done[b].record(down)
        e2e_flops += info.attn_flops
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, dev)
    peak_tf, hbm, peak_src = _peaks()
    fp8 = bool(cfg.get("fp8"))
    peak_kind = "bf16 dense (burst)"
    if fp8:
        # e4m3 tensor peak: the measured bf16 peak times the nominal 4.5 / 2.25 ratio
        peak_tf, peak_kind = 2.0 * peak_tf, "e4m3 dense (burst) = 2 x measured bf16"
    attn_avg = statistics.mean(attn_ms)
    pub_avg = statistics.mean(pub_ms)
    # publish: read every task's bf16 Q/K/V, write Q and the K/V pages in the
    # page dtype, and re-rotate the anchor key (read its unrotated copy, write
    # the page) -- the window shifts every steady round
    page_es = 1 if fp8 else 2
    n_qkv = (S + 1) * NC * 3 * H * D
    pub_bytes = n_qkv * 2 + n_qkv * page_es + 2 * NC * H * D * page_es
    per_launch = flops / args.steps
    achieved = per_launch / (attn_avg * 1e-3) / 1e12
    value = world * flops / (ms * 1e-3) / 1e12
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1)/sqrt(128) Q/K/V, device-resident ring of 3 rounds)",
        "config": {"workload": args.config, "desc": cfg["desc"], "S": S, "chunk_tokens": NC,
                   "heads": H, "head_dim": D, "history_chunks": W, "n_chunks": n_chunks,
                   "rounds": "steady (all S+1 tasks live, anchor re-rotated each round)",
                   "l2": "inputs larger than L2 (K/V pages ~260 MB + Q/K/V 216 MB per round)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "e2e": {"value": round(world * e2e_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
                "d2h_bytes_per_step": host_out[0].numel() * host_out[0].element_size(),
                "ms_per_step": round(e2e_ms / max(1, e2e_steps), 4), "steps": e2e_steps,
                "h2d_link_gbs": {"one_stream": round(link[1], 1), "two_streams": round(link[2], 1)}},
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "tensor", "kernel": "attn_tc_kernel",
                     "achieved": round(achieved, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4),
                     "peak_source": f"{peak_src} {peak_kind}",
                     "avg_launch_ms": round(attn_avg, 4),
                     "flops_per_launch": per_launch,
                     "traffic": attn_traffic("e4m3" if fp8 else "bf16")[0],
                     "traffic_source": attn_traffic("e4m3" if fp8 else "bf16")[1]},
        "publish": {"bound": "hbm", "kernel": "publish_fp8_kernel" if fp8 else "publish_kernel<bf16>",
                    "achieved": round(pub_bytes / (pub_avg * 1e-3) / 1e9, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(pub_bytes / (pub_avg * 1e-3) / 1e9 / hbm, 4),
                    "avg_launch_ms": round(pub_avg, 4), "bytes_per_launch": pub_bytes},
        "clocks": clocks,
    }
    return res


class OracleSample:
    """The oracle (fp64 CPU) on a bounded sample of the steady Wan-shaped
    round (k = S + W + 2): ``rows`` query rows of every task, for the given
    heads.  Inputs are generated in the constructor, before any clock runs;
    ``run`` times only the oracle (RoPE in fp64, materialised mask, dense
    masked softmax attention)."""

    def __init__(self, heads=(0,), seed=5):
        import torch
        import wf_synth
        from oracle import schedule as sch
        from oracle.round import Geom

        cfg_ = CONFIGS["wan13_attn"]
        self.cfg = sch.Cfg(cfg_["S"], 133, cfg_["history"])
        self.geom = Geom(*cfg_["grid"], len(heads), cfg_["head_dim"])
        self.k = self.cfg.S + self.cfg.history + 2
        self.tasks = sch.round_tasks(self.cfg, self.k)
        NC = self.geom.chunk_tokens
        s = 1.0 / math.sqrt(cfg_["head_dim"])
        hs = list(heads)
        self.cache = {}
        for t in self.tasks:
            for key in [(t.chunk, t.stage)] + [(e.chunk, e.j if e.kind == sch.KIND_LIVE else self.cfg.S)
                                               for e in t.context]:
                if key not in self.cache:
                    x = wf_synth.qkv_raw(seed, key[0], key[1], 0, NC, cfg_["heads"],
                                         cfg_["head_dim"], scale=s, dtype=torch.bfloat16)
                    self.cache[key] = x[:, :, hs].double().numpy()

    def run(self, rows):
        """-> (algorithmic FLOPs, seconds) for ``rows`` query rows per task."""
        import numpy as np
        from oracle.round import round_attention

        NC = self.geom.chunk_tokens
        idx = np.linspace(0, NC - 1, rows).astype(int)
        t0 = time.perf_counter()
        round_attention(self.cfg, self.geom, self.k, 0, lambda c, s_, l: self.cache[(c, s_)], rows=idx)
        dt = time.perf_counter() - t0
        fl = sum(4 * rows * len(t.context) * NC * self.geom.head_dim * self.geom.heads
                 for t in self.tasks)
        return fl, dt


def tiny_all_rounds():
    """The fp64 oracle on the tiny fp32 wavefront (S = 2, 6 chunks of 3 x 4 x 4
    tokens, 2 heads x 32, full history): every one of its 8 rounds.
    -> (algorithmic FLOPs, seconds)."""
    import torch
    import wf_synth
    from oracle import schedule as sch
    from oracle.round import Geom, round_attention

    cfg, geom = sch.Cfg(2, 6, -1), Geom(3, 4, 4, 2, 32)
    NC = geom.chunk_tokens
    cache = {}

    def raw(c, s_, l):
        if (c, s_, l) not in cache:
            cache[(c, s_, l)] = wf_synth.qkv_raw(1, c, s_, l, NC, geom.heads, geom.head_dim,
                                                 dtype=torch.float32).double().numpy()
        return cache[(c, s_, l)]

    for k in range(sch.n_rounds(cfg)):          # inputs drawn before the clock runs
        for t in sch.round_tasks(cfg, k):
            raw(t.chunk, t.stage, 0)
    fl = 0.0
    t0 = time.perf_counter()
    for k in range(sch.n_rounds(cfg)):
        round_attention(cfg, geom, k, 0, raw)
        fl += sum(4 * NC * len(t.context) * NC * geom.head_dim * geom.heads
                  for t in sch.round_tasks(cfg, k))
    return fl, time.perf_counter() - t0


class DitBlockSample:
    """The fp64 DiT oracle on one block of one steady round of the
    random-init Wan2.1-1.3B 4-step DiT (4680-token chunks, dim 1536, 12 heads,
    FFN 8960, W = 3; round k = 9 of a 64-chunk request): the QKV projection,
    q/k RMSNorm and RoPE of every chunk the round's attention reads (the 5
    live tasks, the anchor and the 3 history chunks, each over all its 4680
    tokens), then, for ``rows`` sampled query rows of each task, the masked
    attention over the round's key universe and the rest of the block
    (output projection with gated residual, LN, FFN).  Inputs (weights ~ N(0,
    0.02), N(0, 1) residual-stream rows) are drawn in the constructor."""

    def __init__(self, rows=64, seed=9):
        import numpy as np
        import wf_synth
        from oracle import dit
        from oracle import schedule as sch

        self.S, self.W = 4, 3
        self.cfg = sch.Cfg(self.S, 64, self.W)
        self.grid = (3, 30, 52)
        self.dims = dit.Dims(dim=1536, heads=12, head_dim=128, ffn=8960, layers=1)
        params = wf_synth.dit_params(seed, 1536, 8960, 1, 16, 256, std=0.02)
        self.model = dit.Model(self.cfg, self.grid, self.dims, dit.weights_from(params),
                               [1000.0, 750.0, 500.0, 250.0])
        self.k = self.S + self.W + 2
        self.tasks = sch.round_tasks(self.cfg, self.k)
        self.cached = sorted({(e.kind, e.chunk) for t in self.tasks for e in t.context
                              if e.kind in (sch.KIND_ANCHOR, sch.KIND_HISTORY)})
        NC = 4680
        rng = np.random.default_rng(seed)
        self.x = {(t.chunk, t.stage): rng.standard_normal((NC, 1536)) for t in self.tasks}
        self.xc = {c: rng.standard_normal((NC, 1536)) for _, c in self.cached}
        self.rows = np.linspace(0, NC - 1, rows).astype(int)

    def run(self):
        """-> (algorithmic FLOPs, seconds)."""
        import numpy as np
        from oracle import schedule as sch
        from oracle.attention import masked_attention

        m, S, NC, d = self.model, self.S, 4680, self.dims
        t0 = time.perf_counter()
        m.cache = {}
        for _, c in self.cached:                      # store-pass K/V of the cached chunks
            _, kk, vv, kraw = m.qkv(self.xc[c], S, 0, c)
            m.cache[c] = [(kk, vv, kraw)]
        proj = [m.qkv(self.x[(t.chunk, t.stage)], t.stage, 0, t.chunk) for t in self.tasks]
        entries = {}
        for t in self.tasks:
            for e in t.context:
                if e.kind in (sch.KIND_ANCHOR, sch.KIND_HISTORY):
                    entries[(e.kind, e.chunk)] = e
        ks, vs, lab = [], [], []
        for e in sorted(entries.values(), key=lambda e: (e.kind, e.chunk)):
            kk, vv = m.cached_kv(e, 0)
            ks.append(kk)
            vs.append(vv)
            lab.append(np.full(NC, e.j))
        for t, (_, kk, vv, _) in zip(self.tasks, proj):
            ks.append(kk)
            vs.append(vv)
            lab.append(np.full(NC, t.stage))
        K = np.concatenate(ks).transpose(1, 0, 2)
        V = np.concatenate(vs).transpose(1, 0, 2)
        lab = np.concatenate(lab)
        r = self.rows
        for t, (q, _, _, _) in zip(self.tasks, proj):
            mask = np.broadcast_to(sch.sees(self.cfg, t.stage, lab)[None, :], (len(r), lab.shape[0]))
            o = masked_attention(q[r].transpose(1, 0, 2), K, V, mask).transpose(1, 0, 2)
            m.finish_layer(self.x[(t.chunk, t.stage)][r], o, t.stage, 0)
        dt = time.perf_counter() - t0
        n_proj = len(self.cached) + len(self.tasks)
        fl = n_proj * 2.0 * NC * d.dim * 3 * d.dim
        fl += sum(4.0 * len(r) * len(t.context) * NC * d.head_dim * d.heads for t in self.tasks)
        fl += len(self.tasks) * 2.0 * len(r) * (d.dim * d.dim + 2 * d.dim * d.ffn)
        return fl, dt


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(rows=3072, dit_rows=64):
    """The oracle on the host cores, on the samples the measurement plan
    names: the Wan-1.3B attention round (the headline unit), the tiny fp32
    wavefront over all its rounds, and one block of one round of the 1.3B DiT."""
    fl, dt = OracleSample().run(rows)
    fl1, dt1 = tiny_all_rounds()
    blk = DitBlockSample(rows=dit_rows)
    fl3, dt3 = blk.run()
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": _threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle on the steady Wan-1.3B round (k=9): {rows} of 4680 query rows "
                      f"of each of the 5 tasks, 1 of 12 heads, mask materialised; {dt:.1f} s",
            "tiny_all_rounds": {"seconds": round(dt1, 4), "tflops": round(fl1 / dt1 / 1e12, 6),
                                "flops": fl1,
                                "sample": "fp64 oracle on the tiny fp32 wavefront (S=2, 6 chunks of 48 "
                                          "tokens, 2 x 32 heads, full history): all 8 rounds"},
            "dit13_one_block_one_round": {
                "seconds": round(dt3, 3), "tflops": round(fl3 / dt3 / 1e12, 6), "flops": fl3,
                "sample": f"fp64 DiT oracle, one block of one steady round (k=9) of the 1.3B 4-step "
                          f"DiT: QKV + q/k RMSNorm + RoPE of all 9 chunks the round reads (4680 "
                          f"tokens each), masked attention and the rest of the block for {dit_rows} "
                          f"sampled query rows of each of the 5 tasks"}}


def run_reference(args, rows=64):
    o = OracleSample()
    for _ in range(args.warmup):
        o.run(8)
    tot_fl, tot_dt = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = o.run(rows)
        tot_fl += fl
        tot_dt += dt
    v = tot_fl / tot_dt / 1e12
    cfg = CONFIGS[args.config]
    sample = (f"per step: {rows} of 4680 query rows of each of the 5 tasks, 1 of 12 heads, "
              "steady Wan-1.3B round, fp64 oracle, mask materialised")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_dt / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config, "desc": cfg["desc"]},
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": _threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="wan13_attn",
                    choices=sorted(CONFIGS) + sorted(DIT_CONFIGS) + sorted(QKV_ATTN_CONFIGS)
                    + ["streams", "dit_streams", "peaks"])
    ap.add_argument("--no-dit", action="store_true", help="skip the DiT round measurement")
    ap.add_argument("--layers", type=int, default=None,
                    help="DiT configs: override the block count (smaller profiling captures only)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--attn-kernel", default="auto", choices=["auto", "tc", "simt"],
                    help="attention kernel of the attention-layer workload (default: the library's choice)")
    ap.add_argument("--dit-steps", type=int, default=20,
                    help="steady chunks timed per DiT leg of the default line (14B leg: half)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--peak-seconds", type=float, default=4.0,
                    help="--config peaks: seconds of back-to-back launches for the sustained peak (0: burst only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    if args.config == "peaks":
        if rank == 0:
            print(json.dumps(measure_peaks(seconds=args.peak_seconds)), flush=True)
        return
    if args.config in ("streams", "dit_streams"):
        fn = run_streams if args.config == "streams" else run_dit_streams
        d = fn(args, rank, world, steps=args.steps, warmup=args.warmup)
        if rank == 0:
            print(json.dumps(d), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.config in DIT_CONFIGS or args.config in QKV_ATTN_CONFIGS:
        fn = run_dit if args.config in DIT_CONFIGS else run_qkv_attn
        d = fn(args, args.config, rank, world)
        if rank == 0:
            print(json.dumps(d), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    res = run_ours(args, rank, world)
    if not args.no_dit:
        # the other workloads of the measurement plan, each with its clocks and
        # roofline: batched requests (attention layer, then whole DiT rounds),
        # the 1.3B DiT (bf16 and 8-bit), the 5-step long rollout and the
        # 14B-scale QKV + attention stack
        res["streams"] = run_streams(args, rank, world)
        res["dit_streams"] = run_dit_streams(args, rank, world)
        res["dit"] = run_dit(args, "dit13", rank, world, steps=args.dit_steps, warmup=3)
        res["dit_w8a8"] = run_dit(args, "dit13_w8a8", rank, world, steps=args.dit_steps, warmup=3)
        res["dit_s5"] = run_dit(args, "dit13_s5", rank, world, steps=args.dit_steps, warmup=3)
        res["qkv_attn14b"] = run_qkv_attn(args, "qkv_attn14b", rank, world,
                                          steps=max(5, args.dit_steps // 2), warmup=3)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
