"""wf_round_attention_noalloc against wf_round_attention.

Some callers cannot allocate device memory where they launch attention: a
runtime whose memory manager owns every device byte (a caching allocator or
an arena sized at start-up) has no way to hand the library a separate
scratch buffer, and a steady-state serving loop must not call cudaMalloc
because it can synchronise the whole device.  For them the library keeps the
attention kernel's scheduler counters in a fixed device block of its own.
This test runs that entry point twice in a row, in two consecutive rounds,
and checks each output against the regular entry point's output on the same
inputs, within the bf16 tolerance used by the other parity tests (the two
run the same kernel in the same per-unit order, so the outputs are in fact
identical), for bf16 and for 8-bit (e4m3) pages.  A timeout inside that
kernel is recorded in the plan's status word, where wf_sync_status reads it,
and a later call does not clear it.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
from gpu_helpers import fill_qkv, make_round, raw_fn
from oracle import schedule as sch
from oracle.round import Geom

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [wf.WF_BF16, wf.WF_FP8], ids=["bf16", "e4m3"])
def test_noalloc_matches_regular_entry_point_two_calls(dtype):
    cfg = sch.Cfg(4, 12, 3)
    geom = Geom(3, 10, 10, 2, 128)      # 300 tokens: two full key tiles and a ragged one
    scales = (8.0, 8.0) if dtype == wf.WF_FP8 else (1.0, 1.0)
    r = make_round(cfg, geom, dtype, fp8_scales=scales)
    _, traw = raw_fn(31, geom, torch.bfloat16, qk_scale=2.0)
    ref = r.new_out()
    k_first = cfg.S + cfg.history + 2   # steady: all tasks live, anchor re-rotated
    for k in range(k_first + 2):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
        if k < k_first:
            continue
        r.attention(0, ref, wf.WF_ATTN_TC)
        outs = []
        for _ in range(2):
            o = r.new_out().fill_(float("nan"))
            r.attention_noalloc(0, o)
            outs.append(o)
        torch.cuda.synchronize()
        for o in outs:
            for s in range(cfg.S + 1):
                d = (o[s].float() - ref[s].float()).abs() / ref[s].float().abs().clamp(min=1.0)
                assert torch.isfinite(o[s]).all()
                assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3, (k, s)
                assert torch.equal(o[s], ref[s]), (k, s)
    assert r.sync_status() == wf.WF_OK


def test_noalloc_timeout_stays_visible():
    """The status word the kernel writes on a timeout is the plan's: a
    timeout recorded there (here by the bounded-wait self-test) survives a
    following no-alloc call and is then reported and cleared."""
    cfg = sch.Cfg(2, 6, 2)
    geom = Geom(3, 8, 10, 2, 128)
    r = make_round(cfg, geom, wf.WF_BF16)
    _, traw = raw_fn(7, geom, torch.bfloat16)
    out = r.new_out()
    for _ in range(cfg.S + 1):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
        r.attention_noalloc(0, out)
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_OK
    r.selftest_timeout(20000)
    info = r.step()
    r.publish(0, fill_qkv(r, info, traw, 0))
    r.attention_noalloc(0, out)
    assert r.sync_status() == wf.WF_ETIMEOUT
    r.attention_noalloc(0, out)
    assert r.sync_status() == wf.WF_OK


def test_noalloc_rejects_bad_calls():
    cfg = sch.Cfg(2, 4, 1)
    geom = Geom(3, 4, 4, 2, 32)
    r = make_round(cfg, geom, wf.WF_FP32)
    info = r.step()
    out = r.new_out()
    # before this round's publication of layer 0
    assert wf.lib.wf_round_attention_noalloc(r.plan, 0, out.data_ptr(), None) == wf.WF_EORDER
    r.publish(0, fill_qkv(r, info, raw_fn(1, geom, torch.float32)[1], 0))
    # fp32 / head_dim 32 has no tensor-core kernel
    assert wf.lib.wf_round_attention_noalloc(r.plan, 0, out.data_ptr(), None) == wf.WF_EUNSUPPORTED
    assert wf.lib.wf_round_attention_noalloc(r.plan, 1, out.data_ptr(), None) == wf.WF_ERANGE
    assert wf.lib.wf_round_attention_noalloc(None, 0, out.data_ptr(), None) == wf.WF_EINVAL
    torch.cuda.synchronize()
