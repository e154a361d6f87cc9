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
WF_ANCHOR_ADJACENT = 0
WF_ANCHOR_ABSOLUTE = 1
WF_ATTN_AUTO = 0
WF_ATTN_TC = 1
WF_ATTN_SIMT = 2
WF_MAX_STAGES = 8
WF_MAX_CTX = 32
WF_NOALLOC_SCRATCH_BYTES = 256

# every symbol include/wf.h declares
SYMBOLS = ["wf_plan_opts_default", "wf_plan", "wf_plan_buffer_sizes", "wf_bind",
           "wf_round_step", "wf_page_table", "wf_qkv_rope_publish", "wf_round_attention",
           "wf_round_attention_noalloc", "wf_sync_status", "wf_plan_destroy", "wf_strerror"]


class wf_plan_opts(ctypes.Structure):
    _fields_ = [("n_chunks", ctypes.c_int), ("layers", ctypes.c_int), ("grid_t", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int), ("dtype", ctypes.c_int),
                ("use_anchor", ctypes.c_int), ("anchor_mode", ctypes.c_int),
                ("rope_theta", ctypes.c_double)]


class wf_buffer_sizes(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_size_t), ("qbuf", ctypes.c_size_t), ("pool", ctypes.c_size_t),
                ("out", ctypes.c_size_t), ("scratch", ctypes.c_size_t),
                ("n_pages", ctypes.c_int), ("ring_pages", ctypes.c_int)]


_T = WF_MAX_STAGES + 1


class wf_round_info(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int), ("n_tasks", ctypes.c_int), ("store_chunk", ctypes.c_int),
                ("anchor_tpos", ctypes.c_int), ("task_chunk", ctypes.c_int * _T),
                ("task_stage", ctypes.c_int * _T), ("task_ctx", ctypes.c_int * _T),
                ("attn_flops", ctypes.c_double)]


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
        "wf_sync_status": (I, [P, VP]),
        "wf_plan_destroy": (None, [P]),
        "wf_strerror": (ctypes.c_char_p, [I]),
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
                 anchor_mode=WF_ANCHOR_ADJACENT, rope_theta=10000.0, device="cuda",
                 bind=True):
        o = default_opts()
        o.n_chunks, o.layers = n_chunks, layers
        o.grid_t, o.grid_h, o.grid_w = grid
        o.dtype, o.use_anchor, o.anchor_mode, o.rope_theta = dtype, int(use_anchor), anchor_mode, rope_theta
        self.S, self.NC, self.H, self.D = S, chunk_tokens, heads, head_dim
        self.dtype = dtype
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
        import torch
        return torch.bfloat16 if self.dtype == WF_BF16 else torch.float32

    def bind(self, device="cuda"):
        import torch
        es = 2 if self.dtype == WF_BF16 else 4
        s = self.sizes
        self.pool = torch.zeros(s.pool // es, dtype=self.torch_dtype, device=device)
        self.qbuf = torch.zeros(s.qbuf // es, dtype=self.torch_dtype, device=device)
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

    def attention_noalloc(self, layer, out, stream=None):
        """wf_round_attention_noalloc: the tensor-core kernel with its control
        words in the library's static device block (no caller scratch)."""
        check(lib.wf_round_attention_noalloc(self.plan, layer, ctypes.c_void_p(out.data_ptr()),
                                             _stream_handle(stream)), "wf_round_attention_noalloc")

    def sync_status(self, stream=None):
        return lib.wf_sync_status(self.plan, _stream_handle(stream))

    def pool_view(self):
        """The pool as [P][L][2][H][N_C][D]."""
        s = self.sizes
        L = s.pool // (s.n_pages * 2 * self.H * self.NC * self.D * (2 if self.dtype == WF_BF16 else 4))
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
