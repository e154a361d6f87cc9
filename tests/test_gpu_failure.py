"""Failure detection on the GPU without a fault: a bounded wait that nothing
ever completes gives up after its limit, the kernel returns, the plan's
status word reports WF_ETIMEOUT to the host, and the context keeps working
(the same bounded wait guards every barrier of the attention and GEMM
kernels)."""

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
from gpu_helpers import errors, fill_qkv, make_round, raw_fn
from oracle import schedule as sch
from oracle.round import Geom, round_attention

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_survives():
    cfg = sch.Cfg(2, 4, 1)
    geom = Geom(3, 4, 10, 2, 128)            # 120 tokens
    r = make_round(cfg, geom, wf.WF_BF16)
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_OK
    r.selftest_timeout(20000)                 # 20 ms limit
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_ETIMEOUT
    assert r.sync_status() == wf.WF_OK        # read-and-clear
    # the context is intact: a regular round runs and matches the oracle
    raw, traw = raw_fn(3, geom, torch.bfloat16)
    out = r.new_out()
    for k in range(3):
        info = r.step()
        r.publish(0, fill_qkv(r, info, traw, 0))
        r.attention(0, out, wf.WF_ATTN_TC)
    torch.cuda.synchronize()
    assert r.sync_status() == wf.WF_OK
    ref = round_attention(cfg, geom, 2, 0, raw, qk_dtype="bf16")
    for t, o in zip(sch.round_tasks(cfg, 2), ref):
        mx, mean, rel = errors(out[t.stage].float().cpu().numpy(), o)
        assert mx <= 2e-2 and mean <= 2e-3, (mx, mean)
    r.close()


def test_selftest_limit_is_validated():
    cfg = sch.Cfg(2, 4, 1)
    r = make_round(cfg, Geom(3, 4, 10, 2, 128), wf.WF_BF16)
    with pytest.raises(wf.WfError):
        r.selftest_timeout(0)
    with pytest.raises(wf.WfError):
        r.selftest_timeout(5000000)
    r.close()
