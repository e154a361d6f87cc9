"""GPU parity of several requests batched into one round (wf_group_*).

"Wave Forcing" names serving concurrent streams with batching as the next
step (Sec. 8 Future Work; App. E).  A group concatenates the current rounds
of its member requests; each member must get exactly what its own plan
computes.  Checked here: every member's attention output against the fp64
oracle of its own request (members starting at different rounds, so the
batched rounds mix fill, steady state and drain), bit-identity with the
member's own single-plan launches, the visibility fingerprint with a marker
channel per member (a key read from another request shows up as an O(1)
entry in a foreign channel), and the batched QKV projection with the q/k
RMSNorm against per-member projections (bit-identical pages and queries).
Tolerances as in tests/test_gpu_parity.py.
"""

import ctypes

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
import wf_synth
from gpu_helpers import fill_qkv, raw_fn, scaled_errors
from oracle import schedule as sch
from oracle.round import Geom, round_attention

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, BF16_REL = 2e-2, 2e-3, 2e-2
SMALL = Geom(grid_t=3, grid_h=10, grid_w=10, heads=2, head_dim=128)   # 300 tokens: 2 tiles + 44


def make_group(n, cfg, geom, dtype=wf.WF_BF16, fp8_scales=(1.0, 1.0), layers=1):
    return wf.Group(n, cfg.S, geom.chunk_tokens, geom.heads, geom.head_dim, cfg.history,
                    n_chunks=cfg.n_chunks, layers=layers, grid=geom.grid, dtype=dtype,
                    fp8_scales=fp8_scales, use_anchor=cfg.use_anchor, anchor_mode=cfg.anchor_mode,
                    mask=cfg.mask)


def drive(grp, cfg, starts, on_round):
    """Advance member r from global round starts[r] until its request ends;
    on_round(mask, ks, infos) runs the launches of one global round."""
    n = len(starts)
    ks, done = [-1] * n, [False] * n
    total = max(starts) + sch.n_rounds(cfg)
    for g in range(total):
        mask, infos = 0, {}
        for r in range(n):
            if g < starts[r] or done[r]:
                continue
            info = grp.rounds[r].step()
            if info is None:
                done[r] = True
                continue
            ks[r] = info.k
            infos[r] = info
            mask |= 1 << r
        if mask:
            on_round(mask, ks, infos)
    assert all(k == sch.n_rounds(cfg) - 1 for k in ks)


@pytest.mark.parametrize("kernel", [wf.WF_ATTN_TC, wf.WF_ATTN_SIMT])
@pytest.mark.parametrize("starts", [(0, 3), (0, 2, 5)], ids=["two", "three"])
def test_group_requests_match_oracle(starts, kernel):
    cfg = sch.Cfg(4, 8, 2)
    n = len(starts)
    grp = make_group(n, cfg, SMALL)
    raws = [raw_fn(40 + r, SMALL, torch.bfloat16, qk_scale=2.0) for r in range(n)]
    qkv, out, solo = grp.new_qkv(), grp.new_out(), grp.new_out()
    worst = [(0.0, 0.0, 0.0)]

    def on_round(mask, ks, infos):
        for r, info in infos.items():
            fill_qkv(grp.rounds[r], info, raws[r][1], 0, qkv[r])
        grp.publish(mask, 0, qkv)
        out.fill_(float("nan"))
        grp.attention(mask, 0, out, kernel)
        for r in infos:
            grp.rounds[r].attention(0, solo[r], kernel)
        torch.cuda.synchronize()
        for r in range(n):
            if r not in infos:
                assert torch.isnan(out[r]).all()      # not in this round: untouched
                continue
            ref = round_attention(cfg, SMALL, ks[r], 0, raws[r][0], qk_dtype="bf16")
            for t, o in zip(sch.round_tasks(cfg, ks[r]), ref):
                assert torch.equal(out[r][t.stage], solo[r][t.stage]), (r, ks[r], t.stage)
                e = scaled_errors(out[r][t.stage].float().cpu().numpy(), o)
                worst[0] = tuple(max(a, b) for a, b in zip(worst[0], e))

    drive(grp, cfg, starts, on_round)
    mx, mean, rel = worst[0]
    assert mx <= BF16_MAX and mean <= BF16_MEAN and rel <= BF16_REL, (mx, mean, rel)
    assert grp.rounds[0].sync_status() == wf.WF_OK
    grp.close()


@pytest.mark.parametrize("kernel", [wf.WF_ATTN_TC, wf.WF_ATTN_SIMT])
def test_group_visibility_fingerprint(kernel):
    """Q = 0: each query averages V over its visible keys.  V carries a
    one-hot of the producing chunk (channels 0..63), of the producing stage
    (64..) and of the member (100 + r): every query must see exactly its own
    request's context, 1/len(context) per entry, and nothing of the other."""
    cfg = sch.Cfg(3, 7, 1)
    starts = (0, 1, 4)
    n = len(starts)
    grp = make_group(n, cfg, SMALL)
    qkv, out = grp.new_qkv(), grp.new_out()
    D = SMALL.head_dim

    def on_round(mask, ks, infos):
        qkv.zero_()
        for r, info in infos.items():
            for i in range(info.n_tasks):
                c, s = info.task_chunk[i], info.task_stage[i]
                g = torch.Generator().manual_seed(1000 * r + 100 * c + s)
                qkv[r, s, :, 1] = torch.randn(SMALL.chunk_tokens, SMALL.heads, D, generator=g).to(torch.bfloat16)
                qkv[r, s, :, 2, :, c] = 1.0
                qkv[r, s, :, 2, :, 64 + s] = 1.0
                qkv[r, s, :, 2, :, 100 + r] = 1.0
        grp.publish(mask, 0, qkv)
        grp.attention(mask, 0, out, kernel)
        torch.cuda.synchronize()
        for r in infos:
            for t in sch.round_tasks(cfg, ks[r]):
                want = np.zeros(D)
                for e in t.context:
                    st = e.j if e.kind == sch.KIND_LIVE else cfg.S
                    want[e.chunk] += 1.0 / len(t.context)
                    want[64 + st] += 1.0 / len(t.context)
                want[100 + r] = 1.0
                got = out[r][t.stage].float().cpu().numpy()
                assert np.abs(got - want[None, None, :]).max() <= 2e-3, (r, ks[r], t.stage)

    drive(grp, cfg, starts, on_round)
    grp.close()


@pytest.mark.parametrize("fp8", [None, (4.0, 2.0)], ids=["bf16", "e4m3"])
def test_group_projection_norm_equals_members(fp8):
    """One projection GEMM + q/k RMSNorm + publication over the members' rows
    leaves exactly the pages and queries each member's own
    wf_qkv_proj_rope_publish leaves, and the batched attention exactly each
    member's own output (two identical groups, driven batched and per
    member)."""
    cfg = sch.Cfg(4, 7, 2)
    starts = (0, 2)
    n, dim, NC, H = 2, 256, SMALL.chunk_tokens, SMALL.heads
    dtype = wf.WF_FP8 if fp8 else wf.WF_BF16
    a = make_group(n, cfg, SMALL, dtype, fp8 or (1.0, 1.0))
    b = make_group(n, cfg, SMALL, dtype, fp8 or (1.0, 1.0))
    w = wf_synth.normal(wf_synth.key_of(51, 1), (3 * dim, dim), 0.05, torch.bfloat16).cuda()
    bias = wf_synth.normal(wf_synth.key_of(51, 2), (3 * dim,), 0.5, torch.bfloat16).cuda()
    nq = (1 + wf_synth.normal(wf_synth.key_of(51, 3), (dim,), 0.3)).to(torch.bfloat16).cuda()
    nk = (1 + wf_synth.normal(wf_synth.key_of(51, 4), (dim,), 0.3)).to(torch.bfloat16).cuda()
    x = torch.zeros((n, cfg.S + 1, NC, dim), dtype=torch.bfloat16, device="cuda")
    oa, ob = a.new_out(), b.new_out()
    kb = [-1] * n

    def on_round(mask, ks, infos):
        for r, info in infos.items():
            for i in range(info.n_tasks):
                c, s = info.task_chunk[i], info.task_stage[i]
                x[r, s] = wf_synth.normal(wf_synth.key_of(51, 5, r, c, s), (NC, dim), 1.0,
                                          torch.bfloat16).cuda()
            # the twin group's member enters the same round
            assert b.rounds[r].step().k == ks[r]
            kb[r] = ks[r]
        a.publish_proj(mask, 0, x, w, bias, nq, nk)
        a.attention(mask, 0, oa, wf.WF_ATTN_TC)
        for r in infos:
            b.rounds[r].publish_proj(0, x[r], w, bias, nq, nk)
            b.rounds[r].attention(0, ob[r], wf.WF_ATTN_TC)
        torch.cuda.synchronize()
        assert torch.equal(a.pool.view(torch.uint8), b.pool.view(torch.uint8))
        assert torch.equal(a.qbuf.view(torch.uint8), b.qbuf.view(torch.uint8))
        for r in infos:
            for t in sch.round_tasks(cfg, ks[r]):
                assert torch.equal(oa[r][t.stage], ob[r][t.stage]), (r, ks[r], t.stage)

    drive(a, cfg, starts, on_round)
    assert a.rounds[0].sync_status() == wf.WF_OK
    a.close()
    b.close()


def test_group_rejects_bad_calls():
    cfg = sch.Cfg(2, 4, 1)
    grp = make_group(2, cfg, SMALL)
    out, qkv = grp.new_out(), grp.new_qkv()
    fn = wf.lib.wf_group_attention
    # no member has entered a round yet
    assert fn(grp.group, 0b01, 0, out.data_ptr(), wf.WF_ATTN_TC, None) == wf.WF_ENOROUND
    grp.rounds[0].step()
    assert fn(grp.group, 0b01, 0, out.data_ptr(), wf.WF_ATTN_TC, None) == wf.WF_EORDER
    assert fn(grp.group, 0, 0, out.data_ptr(), wf.WF_ATTN_TC, None) == wf.WF_EINVAL      # empty mask
    assert fn(grp.group, 0b100, 0, out.data_ptr(), wf.WF_ATTN_TC, None) == wf.WF_EINVAL  # no member 2
    assert wf.lib.wf_group_publish(grp.group, 0b11, 0, qkv.data_ptr(), None) == wf.WF_ENOROUND
    assert wf.lib.wf_group_publish(grp.group, 0b01, 1, qkv.data_ptr(), None) == wf.WF_ERANGE
    assert wf.lib.wf_group_publish(grp.group, 0b01, 0, qkv.data_ptr(), None) == wf.WF_OK
    assert fn(grp.group, 0b01, 0, out.data_ptr(), wf.WF_ATTN_TC, None) == wf.WF_OK
    torch.cuda.synchronize()
    # shapes must match and the buffers must be consecutive slices
    other = wf.Round(cfg.S, SMALL.chunk_tokens, SMALL.heads, SMALL.head_dim, 2, n_chunks=cfg.n_chunks,
                     grid=SMALL.grid)
    plans = (ctypes.c_void_p * 2)(grp.rounds[0].plan.value, other.plan.value)
    g2 = ctypes.c_void_p()
    assert wf.lib.wf_group_create(plans, 2, ctypes.byref(g2)) == wf.WF_EINVAL     # W differs
    same = wf.Round(cfg.S, SMALL.chunk_tokens, SMALL.heads, SMALL.head_dim, cfg.history,
                    n_chunks=cfg.n_chunks, grid=SMALL.grid)
    plans = (ctypes.c_void_p * 2)(grp.rounds[0].plan.value, same.plan.value)
    assert wf.lib.wf_group_create(plans, 2, ctypes.byref(g2)) == wf.WF_EINVAL     # own buffers
    plans = (ctypes.c_void_p * 2)(grp.rounds[0].plan.value, grp.rounds[0].plan.value)
    assert wf.lib.wf_group_create(plans, 2, ctypes.byref(g2)) == wf.WF_EINVAL     # duplicate
    assert wf.lib.wf_group_create(plans, 9, ctypes.byref(g2)) == wf.WF_ERANGE
    assert grp.rounds[0].sync_status() == wf.WF_OK
    grp.close()
    other.close()
    same.close()
