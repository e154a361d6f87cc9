"""Python binding of libwf.so (the wavefront-round C ABI, include/wf.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  Importing this package
loads the in-tree shared object and fails loudly if it is missing; there is
no fallback of any kind.

``lib`` exposes the C functions under their C names (wf_plan,
wf_round_step, wf_qkv_rope_publish, wf_round_attention, ...).  ``Round`` is
a small convenience owner of a plan plus torch-allocated buffers.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwf.so")

WF_OK = 0
WF_EINVAL = -1
WF_ERANGE = -2
WF_ENOMEM = -3
WF_ECUDA = -4
WF_ETIMEOUT = -5
WF_EDONE = -6
WF_EUNBOUND = -7
WF_ENOROUND = -8
WF_EUNSUPPORTED = -9
WF_EORDER = -10

WF_FP32 = 0
WF_BF16 = 1
WF_FP8 = 2
WF_ANCHOR_ADJACENT = 0
WF_ANCHOR_ABSOLUTE = 1
WF_MASK_WF = 0
WF_MASK_RF = 1
WF_SCHED_WAVEFRONT = 0
WF_SCHED_SEQUENTIAL = 1
WF_MAX_GROUP_PLANS = 8
WF_ATTN_AUTO = 0
WF_ATTN_TC = 1
WF_ATTN_SIMT = 2
WF_EPI_BF16 = 0
WF_EPI_F32 = 1
WF_EPI_GELU_BF16 = 2
WF_EPI_GATED_RESIDUAL = 3
WF_MAX_STAGES = 8
WF_MAX_CTX = 32
WF_NOALLOC_SCRATCH_BYTES = 256

# every symbol include/wf.h declares
SYMBOLS = ["wf_plan_opts_default", "wf_plan", "wf_plan_buffer_sizes", "wf_bind",
           "wf_round_step", "wf_page_table", "wf_qkv_rope_publish", "wf_round_attention",
           "wf_round_attention_noalloc", "wf_round_attention_tasks", "wf_sync_status", "wf_plan_destroy", "wf_strerror",
           "wf_linear", "wf_qkv_proj_rope_publish", "wf_dit_workspace_size", "wf_dit_bind",
           "wf_dit_round", "wf_selftest_timeout", "wf_plan_state_size", "wf_plan_export_state",
           "wf_plan_import_state", "wf_quantize_weight_e4m3", "wf_linear_e4m3",
           "wf_group_create", "wf_group_publish", "wf_group_proj_publish", "wf_group_attention",
           "wf_group_destroy", "wf_group_dit_workspace_size", "wf_group_dit_bind",
           "wf_group_dit_round"]


class wf_plan_opts(ctypes.Structure):
    _fields_ = [("n_chunks", ctypes.c_int), ("layers", ctypes.c_int), ("grid_t", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int), ("dtype", ctypes.c_int),
                ("use_anchor", ctypes.c_int), ("anchor_mode", ctypes.c_int),
                ("rope_theta", ctypes.c_double), ("mask", ctypes.c_int),
                ("schedule", ctypes.c_int), ("fp8_qk_scale", ctypes.c_double),
                ("fp8_v_scale", ctypes.c_double), ("store_extra_history", ctypes.c_int),
                ("rope_split", ctypes.c_int * 3)]


class wf_buffer_sizes(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_size_t), ("qbuf", ctypes.c_size_t), ("pool", ctypes.c_size_t),
                ("out", ctypes.c_size_t), ("scratch", ctypes.c_size_t),
                ("n_pages", ctypes.c_int), ("ring_pages", ctypes.c_int),
                ("qk_norm_tmp", ctypes.c_size_t)]


_T = WF_MAX_STAGES + 1


class wf_round_info(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int), ("n_tasks", ctypes.c_int), ("store_chunk", ctypes.c_int),
                ("anchor_tpos", ctypes.c_int), ("task_chunk", ctypes.c_int * _T),
                ("task_stage", ctypes.c_int * _T), ("task_ctx", ctypes.c_int * _T),
                ("attn_flops", ctypes.c_double)]


class wf_dit_layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("qkv_w", "qkv_b", "o_w", "o_b", "ffn1_w", "ffn1_b",
                                               "ffn2_w", "ffn2_b", "modulation", "norm_q", "norm_k")]


class wf_dit_model(ctypes.Structure):
    _fields_ = [("model_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int), ("channels", ctypes.c_int),
                ("freq_dim", ctypes.c_int), ("shift", ctypes.c_double),
                ("context_noise", ctypes.c_double), ("timesteps", ctypes.c_double * WF_MAX_STAGES)] + \
        [(n, ctypes.c_void_p) for n in ("patch_w", "patch_b", "t1_w", "t1_b", "t2_w", "t2_b", "tp_w",
                                        "tp_b", "head_w", "head_b", "head_mod")] + \
        [("layers", ctypes.POINTER(wf_dit_layer)), ("linear_fp8", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libwf.so is not built ({LIB_PATH}); run "
                          "`python chunk_causal_dit_round_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, VP = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    sig = {
        "wf_plan_opts_default": (None, [ctypes.POINTER(wf_plan_opts)]),
        "wf_plan": (I, [I, I, I, I, I, ctypes.POINTER(wf_plan_opts), ctypes.POINTER(P)]),
        "wf_plan_buffer_sizes": (I, [P, ctypes.POINTER(wf_buffer_sizes)]),
        "wf_bind": (I, [P, VP, VP, VP]),
        "wf_round_step": (I, [P, ctypes.POINTER(wf_round_info)]),
        "wf_page_table": (I, [P, ctypes.POINTER(ctypes.c_int32), I, ctypes.POINTER(I)]),
        "wf_qkv_rope_publish": (I, [P, I, VP, VP]),
        "wf_round_attention": (I, [P, I, VP, I, VP]),
        "wf_round_attention_noalloc": (I, [P, I, VP, VP]),
        "wf_round_attention_tasks": (I, [P, I, VP, I, ctypes.c_uint, VP]),
        "wf_sync_status": (I, [P, VP]),
        "wf_plan_destroy": (None, [P]),
        "wf_strerror": (ctypes.c_char_p, [I]),
        "wf_linear": (I, [P, VP, ctypes.c_longlong, I, I, I, VP, VP, I, I, I, VP, I, VP, I, I, VP]),
        "wf_qkv_proj_rope_publish": (I, [P, I, VP, VP, VP, VP, VP, VP, VP]),
        "wf_dit_workspace_size": (I, [P, I, I, I, I, I, ctypes.POINTER(ctypes.c_size_t)]),
        "wf_dit_bind": (I, [P, ctypes.POINTER(wf_dit_model), VP, VP]),
        "wf_dit_round": (I, [P, VP, VP, VP, VP, VP]),
        "wf_selftest_timeout": (I, [P, ctypes.c_uint, VP]),
        "wf_quantize_weight_e4m3": (I, [P, VP, I, I, VP, VP, VP]),
        "wf_linear_e4m3": (I, [P, VP, ctypes.c_longlong, I, I, I, VP, VP, VP, I, I, I, VP, I, VP, I, I,
                               VP]),
        "wf_plan_state_size": (I, [P, ctypes.POINTER(ctypes.c_size_t)]),
        "wf_plan_export_state": (I, [P, VP, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
        "wf_plan_import_state": (I, [P, VP, ctypes.c_size_t]),
        "wf_group_create": (I, [ctypes.POINTER(P), I, ctypes.POINTER(P)]),
        "wf_group_publish": (I, [P, ctypes.c_uint, I, VP, VP]),
        "wf_group_proj_publish": (I, [P, ctypes.c_uint, I, VP, VP, VP, VP, VP, VP, VP]),
        "wf_group_attention": (I, [P, ctypes.c_uint, I, VP, I, VP]),
        "wf_group_destroy": (None, [P]),
        "wf_group_dit_workspace_size": (I, [P, I, I, I, I, I, ctypes.POINTER(ctypes.c_size_t)]),
        "wf_group_dit_bind": (I, [P, ctypes.POINTER(wf_dit_model), VP, VP]),
        "wf_group_dit_round": (I, [P, ctypes.c_uint, VP, VP, VP, VP, VP]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


class WfError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {lib.wf_strerror(code).decode()} ({code})")


def check(code, what=""):
    if code != WF_OK:
        raise WfError(code, what)
    return code


def default_opts() -> wf_plan_opts:
    o = wf_plan_opts()
    lib.wf_plan_opts_default(ctypes.byref(o))
    return o


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Round:
    """A plan plus its caller-owned device buffers (allocated with torch).

    ``publish(layer, qkv)`` and ``attention(layer, out)`` launch on the given
    (or current) torch stream; ``step()`` advances the round."""

    def __init__(self, S, chunk_tokens, heads, head_dim, history, *, n_chunks, layers=1,
                 grid=(3, 0, 0), dtype=WF_BF16, use_anchor=True,
                 anchor_mode=WF_ANCHOR_ADJACENT, rope_theta=10000.0, mask=WF_MASK_WF,
                 schedule=WF_SCHED_WAVEFRONT, fp8_scales=(1.0, 1.0), store_extra=0, rope_split=None,
                 device="cuda", bind=True):
        o = default_opts()
        o.n_chunks, o.layers = n_chunks, layers
        o.grid_t, o.grid_h, o.grid_w = grid
        o.dtype, o.use_anchor, o.anchor_mode, o.rope_theta = dtype, int(use_anchor), anchor_mode, rope_theta
        o.mask, o.schedule = mask, schedule
        o.fp8_qk_scale, o.fp8_v_scale = fp8_scales
        o.store_extra_history = store_extra
        if rope_split is not None:
            o.rope_split[0], o.rope_split[1], o.rope_split[2] = rope_split
        self.S, self.NC, self.H, self.D = S, chunk_tokens, heads, head_dim
        self.dtype = dtype
        self.n_chunks, self.schedule = n_chunks, schedule
        h = ctypes.c_void_p()
        check(lib.wf_plan(S, chunk_tokens, heads, head_dim, history, ctypes.byref(o),
                          ctypes.byref(h)), "wf_plan")
        self.plan = h
        self.sizes = wf_buffer_sizes()
        check(lib.wf_plan_buffer_sizes(self.plan, ctypes.byref(self.sizes)), "wf_plan_buffer_sizes")
        self.info = None
        if bind:
            self.bind(device)

    @property
    def torch_dtype(self):
        """Element type of the Q/K/V input and the attention output."""
        import torch
        return torch.float32 if self.dtype == WF_FP32 else torch.bfloat16

    @property
    def page_dtype(self):
        """Element type of the query workspace and the K/V pages."""
        import torch
        return torch.float8_e4m3fn if self.dtype == WF_FP8 else self.torch_dtype

    def bind(self, device="cuda", pool=None, qbuf=None):
        """wf_bind to new device buffers, or to the given 1-D ``pool`` /
        ``qbuf`` tensors (slices of a group's allocation)."""
        import torch
        es = {WF_FP32: 4, WF_BF16: 2, WF_FP8: 1}[self.dtype]
        s = self.sizes
        store = torch.uint8 if es == 1 else self.torch_dtype
        self.pool = pool if pool is not None else torch.zeros(s.pool // es, dtype=store, device=device)
        self.qbuf = qbuf if qbuf is not None else torch.zeros(s.qbuf // es, dtype=store, device=device)
        if es == 1:
            self.pool = self.pool.view(self.page_dtype)
            self.qbuf = self.qbuf.view(self.page_dtype)
        self.scratch = torch.zeros(s.scratch, dtype=torch.uint8, device=device)
        check(lib.wf_bind(self.plan, ctypes.c_void_p(self.pool.data_ptr()),
                          ctypes.c_void_p(self.qbuf.data_ptr()),
                          ctypes.c_void_p(self.scratch.data_ptr())), "wf_bind")

    def step(self):
        info = wf_round_info()
        rc = lib.wf_round_step(self.plan, ctypes.byref(info))
        if rc == WF_EDONE:
            return None
        check(rc, "wf_round_step")
        self.info = info
        return info

    def n_left(self):
        """Rounds this request still has after the current one."""
        total = self.n_chunks * (self.S + 1) if self.schedule == WF_SCHED_SEQUENTIAL \
            else self.n_chunks + self.S
        return total - 1 - (self.info.k if self.info is not None else -1)

    def page_table(self):
        cap = 4096
        buf = (ctypes.c_int32 * (10 * cap))()
        n = ctypes.c_int()
        check(lib.wf_page_table(self.plan, buf, cap, ctypes.byref(n)), "wf_page_table")
        rows = [tuple(buf[10 * i:10 * i + 10]) for i in range(n.value)]
        return rows

    def new_qkv(self):
        import torch
        return torch.empty((self.S + 1, self.NC, 3, self.H, self.D), dtype=self.torch_dtype,
                           device=self.pool.device)

    def new_out(self):
        import torch
        return torch.zeros((self.S + 1, self.NC, self.H, self.D), dtype=self.torch_dtype,
                           device=self.pool.device)

    def publish(self, layer, qkv, stream=None):
        check(lib.wf_qkv_rope_publish(self.plan, layer, ctypes.c_void_p(qkv.data_ptr()),
                                      _stream_handle(stream)), "wf_qkv_rope_publish")

    def attention(self, layer, out, kernel=WF_ATTN_AUTO, stream=None):
        check(lib.wf_round_attention(self.plan, layer, ctypes.c_void_p(out.data_ptr()), kernel,
                                     _stream_handle(stream)), "wf_round_attention")

    def attention_tasks(self, layer, out, slot_mask, kernel=WF_ATTN_AUTO, stream=None):
        """wf_round_attention_tasks: the round attention of the active tasks
        whose slot bit is set in slot_mask."""
        check(lib.wf_round_attention_tasks(self.plan, layer, ctypes.c_void_p(out.data_ptr()), kernel,
                                           slot_mask, _stream_handle(stream)),
              "wf_round_attention_tasks")

    def attention_noalloc(self, layer, out, stream=None):
        """wf_round_attention_noalloc: the tensor-core kernel with its control
        words in the library's static device block (no caller scratch)."""
        check(lib.wf_round_attention_noalloc(self.plan, layer, ctypes.c_void_p(out.data_ptr()),
                                             _stream_handle(stream)), "wf_round_attention_noalloc")

    def publish_proj(self, layer, x, w_qkv, b_qkv=None, norm_q=None, norm_k=None, stream=None):
        """wf_qkv_proj_rope_publish: QKV projection of x [S+1, N_C, dim] fused
        with RoPE and paged publication; with the gains norm_q / norm_k the
        q/k RMSNorm runs before RoPE (its q | k workspace is allocated here
        on first use)."""
        tmp = None
        if norm_q is not None:
            import torch
            if getattr(self, "_qk_tmp", None) is None:
                self._qk_tmp = torch.empty(self.sizes.qk_norm_tmp, dtype=torch.uint8,
                                           device=self.pool.device)
            tmp = self._qk_tmp
        check(lib.wf_qkv_proj_rope_publish(self.plan, layer, _ptr(x), _ptr(w_qkv), _ptr(b_qkv),
                                           _ptr(norm_q), _ptr(norm_k), _ptr(tmp),
                                           _stream_handle(stream)), "wf_qkv_proj_rope_publish")

    def linear(self, a, w, bias, out, epilogue, row_begin=0, row_end=None, gate=None,
               rows_per_group=1, stream=None):
        """wf_linear on 2-D tensors: a [rows, K] bf16, w [N, K] bf16."""
        rows, K = a.shape
        N = w.shape[0]
        row_end = rows if row_end is None else row_end
        check(lib.wf_linear(self.plan, _ptr(a), rows, a.stride(0), row_begin, row_end, _ptr(w),
                            _ptr(bias), N, K, epilogue, _ptr(out), out.stride(0), _ptr(gate),
                            gate.stride(0) if gate is not None else 0, rows_per_group,
                            _stream_handle(stream)), "wf_linear")

    def export_state(self) -> bytes:
        """wf_plan_export_state: the host round state as bytes."""
        n = ctypes.c_size_t()
        check(lib.wf_plan_state_size(self.plan, ctypes.byref(n)), "wf_plan_state_size")
        buf = ctypes.create_string_buffer(n.value)
        w = ctypes.c_size_t()
        check(lib.wf_plan_export_state(self.plan, buf, n.value, ctypes.byref(w)),
              "wf_plan_export_state")
        return buf.raw[:w.value]

    def import_state(self, state: bytes):
        check(lib.wf_plan_import_state(self.plan, state, len(state)), "wf_plan_import_state")

    def selftest_timeout(self, limit_us=10000, stream=None):
        check(lib.wf_selftest_timeout(self.plan, limit_us, _stream_handle(stream)),
              "wf_selftest_timeout")

    def quantize_weight_e4m3(self, w, stream=None):
        """wf_quantize_weight_e4m3 on a bf16 [N, K] tensor -> (w8 uint8 [N, K], scale float [N])."""
        import torch
        N, K = w.shape
        w8 = torch.empty((N, K), dtype=torch.uint8, device=w.device)
        sc = torch.empty(N, dtype=torch.float32, device=w.device)
        check(lib.wf_quantize_weight_e4m3(self.plan, _ptr(w), N, K, _ptr(w8), _ptr(sc),
                                          _stream_handle(stream)), "wf_quantize_weight_e4m3")
        return w8, sc

    def linear_e4m3(self, a8, w8, wscale, bias, out, epilogue, row_begin=0, row_end=None,
                    gate=None, rows_per_group=1, stream=None):
        rows, K = a8.shape
        N = w8.shape[0]
        row_end = rows if row_end is None else row_end
        check(lib.wf_linear_e4m3(self.plan, _ptr(a8), rows, a8.stride(0), row_begin, row_end,
                                 _ptr(w8), _ptr(wscale), _ptr(bias), N, K, epilogue, _ptr(out),
                                 out.stride(0), _ptr(gate), gate.stride(0) if gate is not None else 0,
                                 rows_per_group, _stream_handle(stream)), "wf_linear_e4m3")

    def sync_status(self, stream=None):
        return lib.wf_sync_status(self.plan, _stream_handle(stream))

    def pool_view(self):
        """The pool as [P][L][2][H][N_C][D]."""
        s = self.sizes
        es = {WF_FP32: 4, WF_BF16: 2, WF_FP8: 1}[self.dtype]
        L = s.pool // (s.n_pages * 2 * self.H * self.NC * self.D * es)
        return self.pool.view(s.n_pages, L, 2, self.H, self.NC, self.D)

    def close(self):
        if getattr(self, "plan", None):
            lib.wf_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Group:
    """A wf_group over ``n`` plans of one shape: one allocation for their
    pools and query workspaces (sliced per plan), the plans themselves
    (``rounds[r]``, each advanced with its own ``step()``), and the batched
    launches over the members selected by ``mask``."""

    def __init__(self, n, S, chunk_tokens, heads, head_dim, history, device="cuda", **kw):
        import torch
        self.rounds = [Round(S, chunk_tokens, heads, head_dim, history, bind=False, **kw)
                       for _ in range(n)]
        r0 = self.rounds[0]
        es = {WF_FP32: 4, WF_BF16: 2, WF_FP8: 1}[r0.dtype]
        store = torch.uint8 if es == 1 else r0.torch_dtype
        s = r0.sizes
        self.pool = torch.zeros(n * s.pool // es, dtype=store, device=device)
        self.qbuf = torch.zeros(n * s.qbuf // es, dtype=store, device=device)
        for i, r in enumerate(self.rounds):
            r.bind(device, pool=self.pool[i * s.pool // es:(i + 1) * s.pool // es],
                   qbuf=self.qbuf[i * s.qbuf // es:(i + 1) * s.qbuf // es])
        plans = (ctypes.c_void_p * n)(*[r.plan.value for r in self.rounds])
        h = ctypes.c_void_p()
        check(lib.wf_group_create(plans, n, ctypes.byref(h)), "wf_group_create")
        self.group, self.n = h, n
        self.S, self.NC, self.H, self.D = S, chunk_tokens, heads, head_dim
        self._qk_tmp = None

    def new_qkv(self):
        import torch
        r0 = self.rounds[0]
        return torch.zeros((self.n, self.S + 1, self.NC, 3, self.H, self.D), dtype=r0.torch_dtype,
                           device=self.pool.device)

    def new_out(self):
        import torch
        r0 = self.rounds[0]
        return torch.zeros((self.n, self.S + 1, self.NC, self.H, self.D), dtype=r0.torch_dtype,
                           device=self.pool.device)

    def publish(self, mask, layer, qkv, stream=None):
        check(lib.wf_group_publish(self.group, mask, layer, _ptr(qkv), _stream_handle(stream)),
              "wf_group_publish")

    def publish_proj(self, mask, layer, x, w_qkv, b_qkv=None, norm_q=None, norm_k=None, stream=None):
        tmp = None
        if norm_q is not None:
            import torch
            if self._qk_tmp is None:
                self._qk_tmp = torch.empty(self.n * self.rounds[0].sizes.qk_norm_tmp, dtype=torch.uint8,
                                           device=self.pool.device)
            tmp = self._qk_tmp
        check(lib.wf_group_proj_publish(self.group, mask, layer, _ptr(x), _ptr(w_qkv), _ptr(b_qkv),
                                        _ptr(norm_q), _ptr(norm_k), _ptr(tmp), _stream_handle(stream)),
              "wf_group_proj_publish")

    def attention(self, mask, layer, out, kernel=WF_ATTN_AUTO, stream=None):
        check(lib.wf_group_attention(self.group, mask, layer, _ptr(out), kernel, _stream_handle(stream)),
              "wf_group_attention")

    def close(self):
        if getattr(self, "group", None):
            lib.wf_group_destroy(self.group)
            self.group = None
        for r in getattr(self, "rounds", []):
            r.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DitModel:
    """The wf_dit_model of a parameter dict (torch bf16 tensors, copied to
    `dev` and kept alive here)."""

    def __init__(self, dev, dim, params: dict, *, ffn, channels, freq, timesteps, shift,
                 context_noise, linear_fp8):
        self.params = {k: ([t.to(dev).contiguous() for t in v] if isinstance(v, list)
                           else v.to(dev).contiguous()) for k, v in params.items()}
        P = self.params
        L = len(P["qkv_w"])
        m = wf_dit_model()
        m.model_dim, m.ffn_dim, m.channels, m.freq_dim = dim, ffn, channels, freq
        m.shift, m.context_noise = shift, context_noise
        for i, t in enumerate(timesteps):
            m.timesteps[i] = t
        for n in ("patch_w", "patch_b", "t1_w", "t1_b", "t2_w", "t2_b", "tp_w", "tp_b", "head_w",
                  "head_b", "head_mod"):
            setattr(m, n, P[n].data_ptr())
        self._layers = (wf_dit_layer * L)()
        names = [("qkv_w", "qkv_w"), ("qkv_b", "qkv_b"), ("o_w", "o_w"), ("o_b", "o_b"),
                 ("ffn1_w", "f1_w"), ("ffn1_b", "f1_b"), ("ffn2_w", "f2_w"), ("ffn2_b", "f2_b"),
                 ("modulation", "mod"), ("norm_q", "nq"), ("norm_k", "nk")]
        for l in range(L):
            for cn, pn in names:
                setattr(self._layers[l], cn, P[pn][l].data_ptr())
        m.layers = self._layers
        m.linear_fp8 = int(linear_fp8)
        self.model = m
        self.dims = (dim, ffn, channels, freq, int(linear_fp8))


class Dit:
    """A DiT model bound to a Round: device weights (torch bf16 tensors, kept
    alive here), the workspace, and ``round(z_new, eps, x0_out, chunk_out)``
    launching wf_dit_round for the round the plan is in."""

    def __init__(self, rnd: Round, params: dict, *, ffn, channels=16, freq=256, timesteps,
                 shift=5.0, context_noise=0.0, linear_fp8=False, stream=None):
        import torch
        self.r = rnd
        dev = rnd.pool.device
        md = _DitModel(dev, rnd.H * rnd.D, params, ffn=ffn, channels=channels, freq=freq,
                       timesteps=timesteps, shift=shift, context_noise=context_noise,
                       linear_fp8=linear_fp8)
        self._md, self.params, self.model = md, md.params, md.model
        nbytes = ctypes.c_size_t()
        check(lib.wf_dit_workspace_size(rnd.plan, *md.dims, ctypes.byref(nbytes)),
              "wf_dit_workspace_size")
        self.workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        check(lib.wf_dit_bind(rnd.plan, ctypes.byref(md.model), _ptr(self.workspace),
                              _stream_handle(stream)), "wf_dit_bind")

    def round(self, z_new, eps, x0_out=None, chunk_out=None, stream=None):
        check(lib.wf_dit_round(self.r.plan, _ptr(z_new), _ptr(eps), _ptr(x0_out), _ptr(chunk_out),
                               _stream_handle(stream)), "wf_dit_round")


class GroupDit:
    """A DiT model bound to a Group (wf_group_dit_bind); ``round(mask, z_new,
    eps, x0_out, chunk_out)`` runs the DiT round of the selected members, each
    already stepped into its round.  z_new [n][latent], eps [n][S][latent],
    x0_out [n][S+1][latent], chunk_out [n][latent]."""

    def __init__(self, grp: Group, params: dict, *, ffn, channels=16, freq=256, timesteps,
                 shift=5.0, context_noise=0.0, linear_fp8=False, stream=None):
        import torch
        self.g = grp
        dev = grp.pool.device
        md = _DitModel(dev, grp.H * grp.D, params, ffn=ffn, channels=channels, freq=freq,
                       timesteps=timesteps, shift=shift, context_noise=context_noise,
                       linear_fp8=linear_fp8)
        self._md, self.params, self.model = md, md.params, md.model
        nbytes = ctypes.c_size_t()
        check(lib.wf_group_dit_workspace_size(grp.group, *md.dims, ctypes.byref(nbytes)),
              "wf_group_dit_workspace_size")
        self.workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        check(lib.wf_group_dit_bind(grp.group, ctypes.byref(md.model), _ptr(self.workspace),
                                    _stream_handle(stream)), "wf_group_dit_bind")

    def round(self, mask, z_new, eps, x0_out=None, chunk_out=None, stream=None):
        check(lib.wf_group_dit_round(self.g.group, mask, _ptr(z_new), _ptr(eps), _ptr(x0_out),
                                     _ptr(chunk_out), _stream_handle(stream)), "wf_group_dit_round")
