"""The chunk-wise causal DiT forward of one wavefront round, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Wave Forcing" runs, in round k, the forward G_theta of every active task --
chunk k - s at denoising stage s for each active s < S, plus the store pass of
chunk k - S (Sec. 3.1 Eq. 3) -- and then applies the stage transition of
Sec. 2 Eq. 1:

    Z_i^(s+1) = Psi_{nu_{s+1}}( G_theta(Z_i^(s), nu_s | C_{i,s}), eps_{i,s} ),
    Psi_0(x, eps) = x,

where G_theta predicts clean latents and the store pass runs G_theta on the
clean chunk B_i at the context_noise timestep, keeps every layer's K/V and
discards its prediction (Sec. 2; App. B.3).  The model is the standard Wan2.1
transformer (App. D.2: "retain the standard Wan2.1 architectures"); Sec. 4.1
splits one layer into P (QKV projection and RoPE) and C (attention and the
remaining block).  The pages print none of the block's arithmetic, so this
oracle writes the plainest reading of a Wan2.1 block without text
cross-attention (the pages omit text conditioning, Sec. 2), listed here and
in the design notes:

* patch embedding: a (1, 2, 2) patch of C latent channels is a vector of
  4C values ordered (channel, row offset, column offset), mapped to dim by a
  linear layer with bias (a stride-(1,2,2) 3D convolution);
* timestep embedding: t -> [cos(t w_i), sin(t w_i)], w_i = 10000^(-i/half),
  256 values; Linear(256, dim), SiLU, Linear(dim, dim) gives e; SiLU then
  Linear(dim, 6 dim) gives e0;
* block l: (shift_a, scale_a, gate_a, shift_f, scale_f, gate_f) = the six
  rows of m_l + e0 (m_l a learned [6, dim] table);
  x' = LN(x) (1 + scale_a) + shift_a           (LayerNorm eps 1e-6, no affine)
  q, k, v = split(x' W_qkv^T + b_qkv)
  q = RMSNorm(q) g_q, k = RMSNorm(k) g_k   (over the full width dim, all heads
                                           together, eps 1e-6; learned gains)
  RoPE on q and k
  x = x + gate_a * (Attn(q, k, v) W_o^T + b_o)
  x = x + gate_f * (GELU_tanh((LN(x)(1 + scale_f) + shift_f) W_1^T + b_1) W_2^T + b_2)
* head: (shift, scale) = head table [2, dim] + e; y = (LN(x)(1 + scale) +
  shift) W_h^T + b_h, 4C outputs per token ordered (row offset, column
  offset, channel), scattered back to the latent grid;
* timesteps: nu in [0, 1000] is warped with shift 5 (App. A):
  sigma = nu / 1000, sigma' = 5 sigma / (1 + 4 sigma); the model sees
  t = 1000 sigma'; Psi_{nu}(x, eps) = (1 - sigma') x + sigma' eps (flow
  matching; Psi_0 = identity as Eq. 1 requires);
* the store pass uses context_noise = 0 (App. B.3 leaves the value open);
* the q/k normalisation is the standard Wan2.1 block's (App. D.2 keeps that
  architecture): RMSNorm(y) = y / sqrt(mean(y^2) + eps) over the full model
  width, times a learned per-channel gain, applied to the projected q and k
  before RoPE.

``kv_fp8=(qk_scale, v_scale)`` stores the RoPE'd Q and K and V (and the
anchor's unrotated key) as e4m3 after scaling instead of bf16 (8-bit
attention, the pages' SageAttention backend and FP8 K/V payload).

``linear_fp8=True`` runs the block's four linear layers in e4m3 (the pages'
W8A8 backend, Sec. 5): every weight row is scaled by max|w| / 448 (computed
in float32, as the kernel computes it) and rounded to e4m3; the LN outputs,
the attention output and the FFN hidden layer enter those layers as e4m3
with unit scale.

``bf16=True`` rounds to bfloat16 where a BF16 execution (App. B.1) stores a
tensor: the latent patches, every linear layer's input (normalised
activations, attention output, FFN hidden), the projected q and k that the
RMSNorm reads, the RoPE-applied Q/K and V that enter attention (App. B.2
pages), and the weights (given already rounded).
The residual stream, statistics and accumulations stay fp64.

Two formulations of a round (they must agree, App. B.6 Proposition 1):

* ``Model.round``        -- layer-major over all tasks, one attention per
  layer over the round's key universe with the materialised token x token
  mask M[q, x] = 1[j(x) >= s(q)] of Sec. 3.1 Eq. 4;
* ``Model.round_replay`` -- one task at a time (store, then stages S-1 .. 0),
  each a full L-layer forward attending without a mask to the concatenation
  of its ordered context (Eq. 5), reading only K/V already published.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import schedule as sch
from .attention import masked_attention
from .rope import chunk_positions, pair_angles, rotate


# ---- elementwise pieces ------------------------------------------------------

def bf16(x):
    """Round fp64 values to bfloat16 (round to nearest even), back in fp64."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def quantize_rows_e4m3(w):
    """Effective fp64 weight of a per-row e4m3 quantisation: scale = max|w_n|
    / 448 in float32 (1 for an all-zero row), q = e4m3(float32(w) / scale),
    returned as q * scale."""
    from .round import e4m3
    w32 = np.asarray(w, np.float32)
    amax = np.abs(w32).max(axis=1)
    sc = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    q = e4m3((w32 / sc[:, None]).astype(np.float32).astype(np.float64))
    return q * sc.astype(np.float64)[:, None]


def layer_norm(x, eps=1e-6):
    """LayerNorm over the last axis without affine parameters."""
    x = np.asarray(x, np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def rms_norm(x, gain, eps=1e-6):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * np.asarray(gain, np.float64)


def gelu_tanh(x):
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def silu(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def sinusoid(t, n=256):
    """Timestep embedding [cos(t w_i) (i < n/2), sin(t w_i)], w_i = 10000^(-i/(n/2))."""
    half = n // 2
    w = 10000.0 ** (-np.arange(half, dtype=np.float64) / half)
    a = float(t) * w
    return np.concatenate([np.cos(a), np.sin(a)])


def warp_sigma(nu, shift=5.0):
    """sigma' = shift sigma / (1 + (shift - 1) sigma), sigma = nu / 1000 (App. A)."""
    s = float(nu) / 1000.0
    return shift * s / (1.0 + (shift - 1.0) * s)


def psi(x0, eps, nu, shift=5.0):
    """Re-noising Psi_nu(x, eps) = (1 - sigma') x + sigma' eps; Psi_0 = identity (Eq. 1)."""
    s = warp_sigma(nu, shift)
    if s == 0.0:
        return np.array(x0, dtype=np.float64)      # no draw is consumed
    return (1.0 - s) * np.asarray(x0, np.float64) + s * np.asarray(eps, np.float64)


# ---- patches -----------------------------------------------------------------

def patchify(z):
    """Latent chunk z [C, F, 2 gh, 2 gw] -> patch rows [F gh gw, 4 C], tokens
    frame-major then h then w, features ordered (channel, row off, col off)."""
    C, F, Hl, Wl = z.shape
    gh, gw = Hl // 2, Wl // 2
    p = z.reshape(C, F, gh, 2, gw, 2)              # c f h q w r
    p = p.transpose(1, 2, 4, 0, 3, 5)              # f h w c q r
    return p.reshape(F * gh * gw, C * 4)


def unpatchify(y, C, F, gh, gw):
    """Head output rows [F gh gw, 4 C], features ordered (row off, col off,
    channel) -> latent [C, F, 2 gh, 2 gw]."""
    p = np.asarray(y).reshape(F, gh, gw, 2, 2, C)  # f h w q r c
    p = p.transpose(5, 0, 1, 3, 2, 4)              # c f h q w r
    return p.reshape(C, F, 2 * gh, 2 * gw)


# ---- model -------------------------------------------------------------------

@dataclass
class Dims:
    dim: int
    heads: int
    head_dim: int
    ffn: int
    layers: int
    channels: int = 16
    freq: int = 256

    @property
    def patch(self) -> int:
        return 4 * self.channels


@dataclass
class Weights:
    """fp64 copies of the (bf16-valued) parameters; W matrices are [out, in]."""
    patch_w: np.ndarray
    patch_b: np.ndarray
    t1_w: np.ndarray
    t1_b: np.ndarray
    t2_w: np.ndarray
    t2_b: np.ndarray
    tp_w: np.ndarray
    tp_b: np.ndarray
    head_w: np.ndarray
    head_b: np.ndarray
    head_mod: np.ndarray          # [2, dim]
    qkv_w: list = field(default_factory=list)
    qkv_b: list = field(default_factory=list)
    o_w: list = field(default_factory=list)
    o_b: list = field(default_factory=list)
    f1_w: list = field(default_factory=list)
    f1_b: list = field(default_factory=list)
    f2_w: list = field(default_factory=list)
    f2_b: list = field(default_factory=list)
    mod: list = field(default_factory=list)   # [6, dim] per layer
    nq: list = field(default_factory=list)    # [dim] RMSNorm gain of q per layer
    nk: list = field(default_factory=list)    # [dim] RMSNorm gain of k per layer


def time_embedding(w: Weights, t):
    """e [dim] and e0 [6, dim] for model timestep t."""
    e = w.t2_w @ silu(w.t1_w @ sinusoid(t, w.t1_w.shape[1]) + w.t1_b) + w.t2_b
    e0 = w.tp_w @ silu(e) + w.tp_b
    return e, e0.reshape(6, -1)


class Model:
    """One request of the wavefront DiT.  ``round(k, z_new, eps)`` runs round
    k; state (latent slot inputs, K/V of stored chunks) carries over."""

    def __init__(self, cfg: sch.Cfg, grid, dims: Dims, w: Weights, timesteps,
                 shift=5.0, context_noise=0.0, theta=10000.0, bf16_points=True, kv_fp8=None,
                 linear_fp8=False):
        assert len(timesteps) == cfg.S
        self.cfg, self.grid, self.d, self.w = cfg, tuple(grid), dims, w
        self.nu = list(timesteps) + [0.0]          # nu_0 > ... > nu_{S-1} > nu_S = 0
        self.shift, self.theta = shift, theta
        self.rb = bf16 if bf16_points else (lambda x: np.asarray(x, np.float64))
        self.kv_fp8 = kv_fp8
        # inputs and weights of the block's linear layers
        if linear_fp8:
            from .round import e4m3
            self.ra = lambda x: e4m3(x)
            q = quantize_rows_e4m3
            self.lw = {"qkv": [q(a) for a in w.qkv_w], "o": [q(a) for a in w.o_w],
                       "f1": [q(a) for a in w.f1_w], "f2": [q(a) for a in w.f2_w]}
        else:
            self.ra = self.rb
            self.lw = {"qkv": w.qkv_w, "o": w.o_w, "f1": w.f1_w, "f2": w.f2_w}
        # model timestep of each slot: stage s -> warped nu_s; the store -> context_noise
        self.slot_t = [1000.0 * warp_sigma(nu, shift) for nu in timesteps]
        self.slot_t.append(1000.0 * warp_sigma(context_noise, shift))
        self.emb = [time_embedding(w, t) for t in self.slot_t]
        self.latent = {}        # (chunk, stage) -> Z input of that task
        self.cache = {}         # chunk -> per layer (K rotated at own position, V, raw K)
        self.nc = grid[0] * grid[1] * grid[2]

    # -- pieces of one task's forward ------------------------------------------
    def embed(self, z):
        return self.rb(patchify(z)) @ self.w.patch_w.T + self.w.patch_b

    def qkv(self, x, slot, layer, chunk):
        """Projected, normalised, RoPE'd Q, K and V [N_C, H, D] plus the
        unrotated (normalised) K."""
        d, w = self.d, self.w
        m = w.mod[layer] + self.emb[slot][1]
        xa = self.ra(layer_norm(x) * (1.0 + m[1]) + m[0])
        y = xa @ self.lw["qkv"][layer].T + w.qkv_b[layer]
        q, k, v = (y[:, i * d.dim:(i + 1) * d.dim] for i in range(3))
        q = rms_norm(self.rb(q), w.nq[layer])
        k = rms_norm(self.rb(k), w.nk[layer])
        q, k, v = (a.reshape(-1, d.heads, d.head_dim) for a in (q, k, v))
        ang = self.angles(chunk)
        if self.kv_fp8 is not None:
            from .round import e4m3
            sqk, sv = self.kv_fp8
            return (e4m3(rotate(q, ang), sqk), e4m3(rotate(k, ang), sqk), e4m3(v, sv), e4m3(k, sqk))
        return self.rb(rotate(q, ang)), self.rb(rotate(k, ang)), self.rb(v), self.rb(k)

    def angles(self, tpos):
        t, h, ww = chunk_positions(tpos, *self.grid)
        return pair_angles(self.d.head_dim, self.theta, t, h, ww)

    def finish_layer(self, x, o, slot, layer):
        """x + attention output projection, then the FFN half of the block."""
        d, w = self.d, self.w
        m = w.mod[layer] + self.emb[slot][1]
        x = x + m[2] * (self.ra(o.reshape(-1, d.dim)) @ self.lw["o"][layer].T + w.o_b[layer])
        xf = self.ra(layer_norm(x) * (1.0 + m[4]) + m[3])
        hmid = self.ra(gelu_tanh(xf @ self.lw["f1"][layer].T + w.f1_b[layer]))
        return x + m[5] * (hmid @ self.lw["f2"][layer].T + w.f2_b[layer])

    def head(self, x, slot):
        w = self.w
        hm = w.head_mod + self.emb[slot][0][None, :]
        y = self.rb(layer_norm(x) * (1.0 + hm[1]) + hm[0]) @ w.head_w.T + w.head_b
        gh, gw = self.grid[1], self.grid[2]
        return unpatchify(y, self.d.channels, self.grid[0], gh, gw)

    def cached_kv(self, e: sch.Entry, layer):
        k_rot, v, k_raw = self.cache[e.chunk][layer]
        if e.kind == sch.KIND_ANCHOR and e.tpos != e.chunk:
            # once the window has moved, the anchor's key is re-rotated from
            # its stored unrotated copy (App. B.3)
            k = rotate(k_raw, self.angles(e.tpos))
            if self.kv_fp8 is not None:
                from .round import e4m3
                return e4m3(k, self.kv_fp8[0]), v
            return self.rb(k), v
        return k_rot, v

    # -- inputs of a round ---------------------------------------------------------
    def task_input(self, t: sch.Task, z_new):
        if t.stage == 0:
            return np.asarray(z_new, np.float64)
        return self.latent[(t.chunk, t.stage)]

    def transition(self, t: sch.Task, x0, eps):
        """Eq. 1: the next-stage input of a denoising task (stage s < S)."""
        s = t.stage
        z = psi(x0, eps[s], self.nu[s + 1], self.shift)
        self.latent[(t.chunk, s + 1)] = z
        return z

    # -- formulation 1: layer-major, masked -----------------------------------------
    def round(self, k, z_new, eps):
        """Round k.  z_new: Z^(0) of chunk k (used when that chunk exists);
        eps[s]: the draw eps_{k-s, s} of stage s's transition.  Returns
        (x0 per task in slot order, emitted clean chunk or None)."""
        cfg, d = self.cfg, self.d
        tasks = sch.round_tasks(cfg, k)
        xs = [self.embed(self.task_input(t, z_new)) for t in tasks]
        cached = {}
        for t in tasks:
            for e in t.context:
                if e.kind in (sch.KIND_ANCHOR, sch.KIND_HISTORY):
                    cached[(e.kind, e.chunk)] = e
        new_cache = {}
        for layer in range(d.layers):
            proj = [self.qkv(x, t.stage, layer, t.chunk) for x, t in zip(xs, tasks)]
            # key universe: cached entries (label S + 1; S + 2 for history
            # only the store keeps), then every live task (label = stage)
            ks, vs, lab = [], [], []
            for e in sorted(cached.values(), key=lambda e: (e.kind, e.chunk)):
                kk, vv = self.cached_kv(e, layer)
                ks.append(kk)
                vs.append(vv)
                lab.append(np.full(self.nc, e.j))
            for t, (_, kk, vv, _) in zip(tasks, proj):
                ks.append(kk)
                vs.append(vv)
                lab.append(np.full(self.nc, t.stage))
            K = np.concatenate(ks).transpose(1, 0, 2)
            V = np.concatenate(vs).transpose(1, 0, 2)
            lab = np.concatenate(lab)
            for i, t in enumerate(tasks):
                q = proj[i][0]
                mask = np.broadcast_to(sch.sees(cfg, t.stage, lab)[None, :], (self.nc, lab.shape[0]))
                o = masked_attention(q.transpose(1, 0, 2), K, V, mask).transpose(1, 0, 2)
                xs[i] = self.finish_layer(xs[i], o, t.stage, layer)
                if t.stage == cfg.S:
                    new_cache.setdefault(t.chunk, []).append((proj[i][1], proj[i][2], proj[i][3]))
        return self._end_round(tasks, xs, eps, new_cache)

    # -- formulation 2: task at a time, ordered contexts ---------------------------
    def round_replay(self, k, z_new, eps):
        cfg, d = self.cfg, self.d
        tasks = sch.round_tasks(cfg, k)
        published = {}     # (chunk, stage) -> per layer (K, V)
        xs = {}
        new_cache = {}
        for t in sorted(tasks, key=lambda t: -t.stage):
            x = self.embed(self.task_input(t, z_new))
            for layer in range(d.layers):
                q, kk, vv, kraw = self.qkv(x, t.stage, layer, t.chunk)
                published.setdefault((t.chunk, t.stage), []).append((kk, vv))
                if t.stage == cfg.S:
                    new_cache.setdefault(t.chunk, []).append((kk, vv, kraw))
                ks, vs = [], []
                for e in t.context:
                    if e.kind in (sch.KIND_STORE, sch.KIND_LIVE):
                        kv = published.get((e.chunk, e.j))
                        if kv is None or len(kv) <= layer:
                            raise AssertionError(f"task {(t.chunk, t.stage)} reads unpublished {(e.chunk, e.j)}")
                        ke, ve = kv[layer]
                    else:
                        ke, ve = self.cached_kv(e, layer)
                    ks.append(ke)
                    vs.append(ve)
                K = np.concatenate(ks).transpose(1, 0, 2)
                V = np.concatenate(vs).transpose(1, 0, 2)
                full = np.ones((self.nc, K.shape[1]), dtype=bool)
                o = masked_attention(q.transpose(1, 0, 2), K, V, full).transpose(1, 0, 2)
                x = self.finish_layer(x, o, t.stage, layer)
            xs[(t.chunk, t.stage)] = x
        return self._end_round(tasks, [xs[(t.chunk, t.stage)] for t in tasks], eps, new_cache)

    def _end_round(self, tasks, xs, eps, new_cache):
        cfg = self.cfg
        x0s, emitted = [], None
        for t, x in zip(tasks, xs):
            x0 = self.head(x, t.stage)
            x0s.append(x0)
            if t.stage < cfg.S:
                z = self.transition(t, x0, eps)
                if t.stage == cfg.S - 1:
                    emitted = z          # B_i = Z_i^(S): Psi_0 is the identity
            self.latent.pop((t.chunk, t.stage), None)
        for c, per_layer in new_cache.items():
            self.cache[c] = per_layer
        return x0s, emitted


def weights_from(params: dict) -> Weights:
    """fp64 copies of a parameter dict (torch tensors, see ``wf_synth.dit_params``)."""
    f = lambda t: t.double().numpy()
    w = Weights(**{k: f(params[k]) for k in ("patch_w", "patch_b", "t1_w", "t1_b", "t2_w",
                                             "t2_b", "tp_w", "tp_b", "head_w", "head_b",
                                             "head_mod")})
    for k in ("qkv_w", "qkv_b", "o_w", "o_b", "f1_w", "f1_b", "f2_w", "f2_b", "mod", "nq", "nk"):
        setattr(w, k, [f(t) for t in params[k]])
    return w
