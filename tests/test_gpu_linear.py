"""GPU parity of the tensor-core linear layers (wf_linear) against fp64 on
the same bf16 operands: plain bf16 / f32 outputs, the GELU hidden layer and
the gated residual add of the DiT block ("Wave Forcing" Sec. 4.1, the
remaining block of a Wan2.1 transformer layer)."""

import ctypes

import numpy as np
import pytest
import torch

import chunk_causal_dit_round_b300 as wf
import wf_synth
from oracle import dit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    r = wf.Round(1, 48, 1, 128, -1, n_chunks=1, grid=(3, 4, 4), dtype=wf.WF_BF16)
    yield r
    r.close()


def operands(seed, M, N, K, rows_extra=0):
    a = wf_synth.normal(wf_synth.key_of(seed, 1), (M + rows_extra, K), 1.0, torch.bfloat16)
    w = wf_synth.normal(wf_synth.key_of(seed, 2), (N, K), 0.05, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(seed, 3), (N,), 0.5, torch.bfloat16)
    return a, w, b


def ref_linear(a, w, b, r0, r1):
    return a[r0:r1].double().numpy() @ w.double().numpy().T + b.double().numpy()


def tol_f32(K):
    # fp32 accumulation of K products of O(1) terms: far below bf16 resolution
    return 1e-4 * np.sqrt(K)


# M spans several 128-row tiles with a ragged tail; N several 256-column tiles
# plus a ragged 32-column remainder; K one and several 64-wide slices.
SHAPES = [(300, 544, 64), (517, 256, 1536), (129, 800, 320), (1, 32, 128)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_f32_epilogue(plan, M, N, K):
    a, w, b = operands(1, M, N, K)
    out = torch.full((M, N), float("nan"), device="cuda")
    plan.linear(a.cuda(), w.cuda(), b.cuda(), out, wf.WF_EPI_F32)
    torch.cuda.synchronize()
    ref = ref_linear(a, w, b, 0, M)
    err = np.abs(out.cpu().double().numpy() - ref).max()
    assert err <= tol_f32(K), err
    assert plan.sync_status() == wf.WF_OK


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_bf16_and_gelu_epilogues(plan, M, N, K):
    a, w, b = operands(2, M, N, K)
    ref = ref_linear(a, w, b, 0, M)
    for epi, fn in ((wf.WF_EPI_BF16, lambda x: x), (wf.WF_EPI_GELU_BF16, dit.gelu_tanh)):
        out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        plan.linear(a.cuda(), w.cuda(), b.cuda(), out, epi)
        torch.cuda.synchronize()
        got = out.cpu().double().numpy()
        want = fn(ref)
        # one bf16 rounding of the result: half an ulp, 2^-9 relative, plus fp32 noise
        err = np.abs(got - want) / np.maximum(np.abs(want), 1e-2)
        assert err.max() <= 2 ** -8, (epi, err.max())


@pytest.mark.parametrize("M,N,K,r0,r1", [(300, 544, 128, 37, 261), (517, 800, 384, 129, 390)])
def test_staged_outputs_row_range(plan, M, N, K, r0, r1):
    """Row-major outputs leave through shared memory and TMA stores in
    32-row x 128-byte blocks: rows [r0, r1) that start and end inside a
    tile, and a ragged last column block, are written; every other row keeps
    its sentinel bit for bit (bf16, GELU bf16, and bf16 out of e4m3
    operands; K a multiple of 128, the e4m3 GEMM's K step)."""
    a, w, b = operands(4, M, N, K)
    ref = ref_linear(a, w, b, r0, r1)
    sentinel = 7.0
    for epi, fn in ((wf.WF_EPI_BF16, lambda x: x), (wf.WF_EPI_GELU_BF16, dit.gelu_tanh)):
        out = torch.full((M, N), sentinel, dtype=torch.bfloat16, device="cuda")
        plan.linear(a.cuda(), w.cuda(), b.cuda(), out, epi, row_begin=r0, row_end=r1)
        torch.cuda.synchronize()
        got = out.cpu().double().numpy()
        assert np.all(got[:r0] == sentinel) and np.all(got[r1:] == sentinel), epi
        want = fn(ref)
        err = np.abs(got[r0:r1] - want) / np.maximum(np.abs(want), 1e-2)
        assert err.max() <= 2 ** -8, (epi, err.max())
    a8 = a.float().to(torch.float8_e4m3fn)
    w8, sc = plan.quantize_weight_e4m3(w.cuda())
    deq_w = w8.cpu().view(torch.float8_e4m3fn).double().numpy() * sc.cpu().double().numpy()[:, None]
    ref8 = a8[r0:r1].double().numpy() @ deq_w.T + b.double().numpy()
    out = torch.full((M, N), sentinel, dtype=torch.bfloat16, device="cuda")
    plan.linear_e4m3(a8.view(torch.uint8).cuda(), w8, sc, b.cuda(), out, wf.WF_EPI_BF16,
                     row_begin=r0, row_end=r1)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    assert np.all(got[:r0] == sentinel) and np.all(got[r1:] == sentinel)
    err = np.abs(got[r0:r1] - ref8) / np.maximum(np.abs(ref8), 1e-2)
    assert err.max() <= 2 ** -8, err.max()
    assert plan.sync_status() == wf.WF_OK


def test_row_range_and_gated_residual(plan):
    """Rows outside [row_begin, row_end) are untouched; row r is gated by
    gate[r // rows_per_group]."""
    M, N, K, G = 3 * 100, 512, 256, 100
    a, w, b = operands(3, M, N, K)
    gate = wf_synth.normal(wf_synth.key_of(3, 9), (3, N), 1.0, torch.float32)
    x0 = wf_synth.normal(wf_synth.key_of(3, 10), (M, N), 1.0, torch.float32)
    out = x0.clone().cuda()
    plan.linear(a.cuda(), w.cuda(), b.cuda(), out, wf.WF_EPI_GATED_RESIDUAL, row_begin=100,
                row_end=300, gate=gate.cuda(), rows_per_group=G)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    ref = x0.double().numpy().copy()
    y = ref_linear(a, w, b, 100, 300)
    g = gate.double().numpy()
    ref[100:300] += g[np.arange(100, 300) // G] * y
    assert np.array_equal(got[:100], x0.double().numpy()[:100])
    assert np.abs(got - ref).max() <= 3 * tol_f32(K)


@pytest.mark.parametrize("M,N,K,r0,r1,G", [
    (300, 800, 192, 37, 300, 7),        # ragged 32-column remainder, groups smaller than a warp
    (517, 256, 1536, 129, 390, 200),    # row range starting inside a tile, ragged last tile
    (64, 1536, 64, 0, 1, 1),            # a single row
])
def test_gated_residual_ranges(plan, M, N, K, r0, r1, G):
    """x += gate[row // G] * (A W^T + b) on rows [r0, r1) only, through the
    reduce-add epilogue; every other element of x keeps its bits."""
    a, w, b = operands(11, M, N, K)
    n_groups = (M + G - 1) // G
    gate = wf_synth.normal(wf_synth.key_of(11, 9), (n_groups, N), 1.0, torch.float32)
    x0 = wf_synth.normal(wf_synth.key_of(11, 10), (M, N), 1.0, torch.float32)
    out = x0.clone().cuda()
    plan.linear(a.cuda(), w.cuda(), b.cuda(), out, wf.WF_EPI_GATED_RESIDUAL, row_begin=r0,
                row_end=r1, gate=gate.cuda(), rows_per_group=G)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    ref = x0.double().numpy().copy()
    ref[r0:r1] += gate.double().numpy()[np.arange(r0, r1) // G] * ref_linear(a, w, b, r0, r1)
    keep = np.ones(M, dtype=bool)
    keep[r0:r1] = False
    assert np.array_equal(got[keep], x0.double().numpy()[keep])
    assert np.abs(got - ref).max() <= 3 * tol_f32(K)
    assert plan.sync_status() == wf.WF_OK


def test_no_bias(plan):
    M, N, K = 200, 256, 128
    a, w, _ = operands(4, M, N, K)
    out = torch.zeros((M, N), device="cuda")
    plan.linear(a.cuda(), w.cuda(), None, out, wf.WF_EPI_F32)
    torch.cuda.synchronize()
    ref = a.double().numpy() @ w.double().numpy().T
    assert np.abs(out.cpu().double().numpy() - ref).max() <= tol_f32(K)


# ---- 8-bit linear layers ----------------------------------------------------------

def e4m3_bytes_np(x32):
    """float32 values -> e4m3 bytes (round to nearest even, saturating)."""
    t = torch.from_numpy(np.clip(x32, -448.0, 448.0).astype(np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_weight_quantisation_bit_exact(plan):
    N, K = 300, 384
    w = wf_synth.normal(wf_synth.key_of(8, 1), (N, K), 0.02, torch.bfloat16)
    w[7].zero_()                                     # an all-zero row keeps scale 1
    w8, sc = plan.quantize_weight_e4m3(w.cuda())
    torch.cuda.synchronize()
    wf32 = w.float().numpy()
    amax = np.abs(wf32).max(axis=1)
    want_sc = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    assert np.array_equal(sc.cpu().numpy(), want_sc)
    q = (wf32 / want_sc[:, None]).astype(np.float32)      # IEEE fp32 division, as the kernel
    assert np.array_equal(w8.cpu().numpy(), e4m3_bytes_np(q))


@pytest.mark.parametrize("M,N,K", [(300, 544, 128), (517, 256, 1536), (129, 800, 384)])
def test_e4m3_linear_epilogues(plan, M, N, K):
    a = wf_synth.normal(wf_synth.key_of(9, 1), (M, K), 1.0, torch.float32)
    a8 = a.to(torch.float8_e4m3fn)
    w = wf_synth.normal(wf_synth.key_of(9, 2), (N, K), 0.05, torch.bfloat16)
    b = wf_synth.normal(wf_synth.key_of(9, 3), (N,), 0.5, torch.bfloat16)
    w8, sc = plan.quantize_weight_e4m3(w.cuda())
    deq_w = w8.cpu().view(torch.float8_e4m3fn).double().numpy() * sc.cpu().double().numpy()[:, None]
    ref = a8.double().numpy() @ deq_w.T + b.double().numpy()
    a8d = a8.view(torch.uint8).cuda()
    out = torch.zeros((M, N), device="cuda")
    plan.linear_e4m3(a8d, w8, sc, b.cuda(), out, wf.WF_EPI_F32)
    torch.cuda.synchronize()
    err = np.abs(out.cpu().double().numpy() - ref).max()
    assert err <= 1e-4 * np.sqrt(K) * max(1.0, np.abs(ref).max()), err
    gate = wf_synth.normal(wf_synth.key_of(9, 4), ((M + 199) // 200, N), 1.0, torch.float32)
    x0 = wf_synth.normal(wf_synth.key_of(9, 5), (M, N), 1.0, torch.float32)
    x = x0.clone().cuda()
    plan.linear_e4m3(a8d, w8, sc, b.cuda(), x, wf.WF_EPI_GATED_RESIDUAL, gate=gate.cuda(),
                     rows_per_group=200)
    torch.cuda.synchronize()
    want = x0.double().numpy() + gate.double().numpy()[np.arange(M) // 200] * ref
    assert np.abs(x.cpu().double().numpy() - want).max() <= 3e-4 * np.sqrt(K) * max(1.0, np.abs(ref).max())
    assert plan.sync_status() == wf.WF_OK


def test_argument_checks_reject_before_launch(plan):
    """Arguments wf_linear cannot serve are rejected with an error code and
    launch nothing: a gated residual without a gate or with rows_per_group 0,
    a misaligned output pitch, rows outside A, K not a multiple of 64."""
    M, N, K = 256, 256, 128
    a, w, b = (t.cuda() for t in operands(12, M, N, K))
    out = torch.zeros((M, N), device="cuda")
    gate = torch.ones((2, N), device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    lib, h = wf.lib, plan.plan

    def call(row_begin=0, row_end=M, epi=wf.WF_EPI_GATED_RESIDUAL, g=gate, g_ld=N, rpg=200, ldo=N,
             k=K, a_rows=M):
        return lib.wf_linear(h, P(a), a_rows, K, row_begin, row_end, P(w), P(b), N, k, epi, P(out), ldo,
                             P(g), g_ld, rpg, None)

    x0 = out.clone()
    assert call(g=None) == wf.WF_EINVAL
    assert call(rpg=0) == wf.WF_EINVAL
    assert call(g_ld=N - 4) == wf.WF_EINVAL
    assert call(ldo=N + 4) == wf.WF_EINVAL                 # pitch not a multiple of 8
    assert call(row_end=M + 1) == wf.WF_ERANGE
    assert call(row_begin=5, row_end=5) == wf.WF_ERANGE
    assert call(k=96) == wf.WF_EINVAL
    assert call(epi=99) == wf.WF_EINVAL
    assert lib.wf_linear_e4m3(h, P(a), M, K, 0, M, P(w), None, P(b), N, K, wf.WF_EPI_F32, P(out), N,
                              None, 0, 1, None) == wf.WF_EINVAL    # no weight scales
    torch.cuda.synchronize()
    assert torch.equal(out, x0)
    assert plan.sync_status() == wf.WF_OK
