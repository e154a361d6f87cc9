"""Derivation of the parity bars of the Wan-width DiT request
(tests/test_gpu_dit.py::test_dit_request_wan_width).  Not collected by
pytest (a CPU run takes a few minutes); run it by hand:

    python tests/derive_wan_width_bars.py

It runs the fp64 DiT oracle on the request the GPU test uses (S = 4, 6
chunks, W = 3, dim 1536, 12 heads x 128, FFN 8960, two blocks, weights
~ N(0, 0.02), 3 x 8 x 10 patches) three times: with the bf16 rounding points
of a BF16 execution, without them (pure fp64), and with the rounding points
plus a planted mask mistake (every query also sees the noisier live chunks,
the reverse edges the chunk-causal mask removes).  It prints the worst
(max, mean, relative L2) of O / max(1, |O|) over every prediction and
emitted chunk for (a) rounding alone and (b) the planted mistake.  The bars
must sit above (a) and at least 3x below (b).  Calls only oracle/ and the
seeded generators."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import wf_synth                                    # noqa: E402
import oracle.dit as od                            # noqa: E402
from oracle import dit                             # noqa: E402
from oracle import schedule as sch                 # noqa: E402
from gpu_helpers import scaled_errors              # noqa: E402


def main():
    cfg = sch.Cfg(4, 6, 3)
    grid = (3, 8, 10)
    dims = dit.Dims(dim=1536, heads=12, head_dim=128, ffn=8960, layers=2, channels=16, freq=256)
    seed = 18
    params = wf_synth.dit_params(seed, dims.dim, dims.ffn, dims.layers, dims.channels, dims.freq,
                                 std=0.02)

    def lat(c, s):
        return wf_synth.latent(seed, c, s, 16, 3, 16, 20).double().numpy()

    def run(b16):
        m = dit.Model(cfg, grid, dims, dit.weights_from(params), [1000.0, 750.0, 500.0, 250.0],
                      bf16_points=b16)
        outs = []
        for k in range(sch.n_rounds(cfg)):
            x0, em = m.round(k, lat(k, -1), [lat(k - s, s) for s in range(4)])
            outs += x0 + ([em] if em is not None else [])
        return outs

    def worst(a, b):
        w = [0.0, 0.0, 0.0]
        for u, v in zip(a, b):
            w = [max(p, q) for p, q in zip(w, scaled_errors(u, v))]
        return w

    ref = run(True)
    print("rounding alone (max, mean, rel):", worst(ref, run(False)))
    orig = od.masked_attention
    try:
        od.masked_attention = lambda q, k, v, mask: orig(q, k, v, np.ones_like(mask))
        print("planted mask mistake (max, mean, rel):", worst(ref, run(True)))
    finally:
        od.masked_attention = orig


if __name__ == "__main__":
    main()
