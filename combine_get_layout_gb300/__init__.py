"""Python binding of libep_gb300.so (MoE dispatch / combine layout on GB300).

Two layers, both argument marshalling only -- every step of layout, dispatch
and combine runs in the library's CUDA kernels:

* ``ep_*`` functions with the C ABI's names and arguments (include/ep.h),
  taking ``EpConfig`` / ``EpLayout`` ctypes structures and raw pointers.
* A torch layer (``Config``, ``Layout``, ``get_layout``, ``dispatch``,
  ``combine``) that allocates device buffers with torch, passes
  ``tensor.data_ptr()`` and the current CUDA stream, and raises ``EpError``
  on a non-zero status.  torch provides memory and streams, nothing else.

There is no fallback: if the shared library is missing, importing this
package raises.  Build it with ``python combine_get_layout_gb300/build_lib.py``.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_EXPERT_RANGE = 2
EP_ERR_DUP_EXPERT = 3
EP_ERR_CAPACITY = 4
EP_ERR_CUDA = 5
EP_ERR_TIMEOUT = 6
EP_ERR_TIMEOUT_PENDING = 7

# The entry points include/ep.h declares (kept in sync by a test).
ABI_SYMBOLS = (
    "ep_recv_capacity",
    "ep_layout_workspace_bytes",
    "ep_get_layout",
    "ep_dispatch",
    "ep_combine",
    "ep_layout_and_dispatch",
    "ep_scale_ld",
    "ep_dispatch_fp8",
    "ep_combine_epilogue",
    "ep_dispatch_backward",
    "ep_combine_backward",
    "ep_rank_rows_capacity",
    "ep_dispatch_ranks",
    "ep_expand",
    "ep_reduce_ranks",
    "ep_combine_ranks",
    "ep_dispatch_from_host",
    "ep_combine_to_host",
    "ep_check_error",
    "ep_selftest_wait_timeout",
    "ep_selftest_layout_timeout",
    "ep_selftest_fp8_quotient",
    "ep_last_cuda_error",
    "ep_get_layout_noalloc",
    "ep_status_str",
)


class EpConfig(ctypes.Structure):
    _fields_ = [
        ("max_tokens", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("num_topk", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("num_ranks", ctypes.c_int32),
        ("expert_alignment", ctypes.c_int32),
        ("use_fp8_dispatch", ctypes.c_int32),
        ("zero_padding", ctypes.c_int32),
    ]


class EpLayout(ctypes.Structure):
    _fields_ = [
        ("expert_count", ctypes.c_void_p),
        ("expert_start", ctypes.c_void_p),
        ("expert_end", ctypes.c_void_p),
        ("rank_start", ctypes.c_void_p),
        ("tokens_per_rank", ctypes.c_void_p),
        ("is_token_in_rank", ctypes.c_void_p),
        ("slot_of", ctypes.c_void_p),
        ("src_info", ctypes.c_void_p),
        ("err", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("rank_row_start", ctypes.c_void_p),
        ("rank_slot_of", ctypes.c_void_p),
        ("rank_src", ctypes.c_void_p),
        ("num_tokens", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python combine_get_layout_gb300/build_lib.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.ep_recv_capacity.restype = i64
    L.ep_recv_capacity.argtypes = [P(EpConfig)]
    L.ep_layout_workspace_bytes.restype = i64
    L.ep_layout_workspace_bytes.argtypes = [P(EpConfig)]
    L.ep_get_layout.restype = i32
    L.ep_get_layout.argtypes = [P(EpConfig), i32, vp, P(EpLayout), vp, vp]
    L.ep_dispatch.restype = i32
    L.ep_dispatch.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp]
    L.ep_combine.restype = i32
    L.ep_combine.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp]
    L.ep_scale_ld.restype = i64
    L.ep_scale_ld.argtypes = [P(EpConfig)]
    L.ep_dispatch_fp8.restype = i32
    L.ep_dispatch_fp8.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp, i32, vp, vp]
    L.ep_combine_epilogue.restype = i32
    L.ep_combine_epilogue.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp, vp, vp]
    L.ep_dispatch_backward.restype = i32
    L.ep_dispatch_backward.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp]
    L.ep_combine_backward.restype = i32
    L.ep_combine_backward.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp]
    L.ep_rank_rows_capacity.restype = i64
    L.ep_rank_rows_capacity.argtypes = [P(EpConfig)]
    L.ep_dispatch_ranks.restype = i32
    L.ep_dispatch_ranks.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp, vp]
    L.ep_expand.restype = i32
    L.ep_expand.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp]
    L.ep_reduce_ranks.restype = i32
    L.ep_reduce_ranks.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp]
    L.ep_combine_ranks.restype = i32
    L.ep_combine_ranks.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp]
    L.ep_layout_and_dispatch.restype = i32
    L.ep_layout_and_dispatch.argtypes = [P(EpConfig), i32, vp, P(EpLayout), vp, vp, vp, vp,
                                         vp, vp]
    L.ep_dispatch_from_host.restype = i32
    L.ep_dispatch_from_host.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, vp, vp,
                                        i32, vp]
    L.ep_combine_to_host.restype = i32
    L.ep_combine_to_host.argtypes = [P(EpConfig), P(EpLayout), vp, vp, vp, vp, i32, vp]
    L.ep_check_error.restype = i32
    L.ep_check_error.argtypes = [P(EpLayout), vp]
    L.ep_selftest_fp8_quotient.restype = i32
    L.ep_selftest_fp8_quotient.argtypes = [vp, vp, vp]
    L.ep_selftest_wait_timeout.restype = i32
    L.ep_selftest_wait_timeout.argtypes = [i64, vp, vp]
    L.ep_selftest_layout_timeout.restype = i32
    L.ep_selftest_layout_timeout.argtypes = [P(EpConfig), i32, vp, P(EpLayout), i32, i64, vp]
    L.ep_get_layout_noalloc.restype = i32
    L.ep_get_layout_noalloc.argtypes = [P(EpConfig), i32, vp, P(EpLayout), vp, vp]
    L.ep_last_cuda_error.restype = i32
    L.ep_last_cuda_error.argtypes = []
    L.ep_status_str.restype = ctypes.c_char_p
    L.ep_status_str.argtypes = [i32]
    return L


_lib = _load()


def lib():
    """The loaded ctypes library (for tests that call the ABI directly)."""
    return _lib


# ---- C-ABI names ------------------------------------------------------------

def ep_recv_capacity(cfg: EpConfig) -> int:
    return int(_lib.ep_recv_capacity(ctypes.byref(cfg)))


def ep_layout_workspace_bytes(cfg: EpConfig) -> int:
    return int(_lib.ep_layout_workspace_bytes(ctypes.byref(cfg)))


def ep_get_layout(cfg, num_tokens, d_topk_idx, layout, h_expert_count, stream) -> int:
    return int(_lib.ep_get_layout(ctypes.byref(cfg), num_tokens, d_topk_idx,
                                  ctypes.byref(layout), h_expert_count, stream))


def ep_dispatch(cfg, layout, d_x, d_topk_weights, d_recv_x, d_recv_scale,
                d_recv_w, stream) -> int:
    return int(_lib.ep_dispatch(ctypes.byref(cfg), ctypes.byref(layout), d_x,
                                d_topk_weights, d_recv_x, d_recv_scale,
                                d_recv_w, stream))


def ep_combine(cfg, layout, d_expert_out, d_topk_weights, d_y, stream) -> int:
    return int(_lib.ep_combine(ctypes.byref(cfg), ctypes.byref(layout),
                               d_expert_out, d_topk_weights, d_y, stream))


def ep_scale_ld(cfg: EpConfig) -> int:
    return int(_lib.ep_scale_ld(ctypes.byref(cfg)))


def ep_dispatch_fp8(cfg, layout, d_x, d_x_q, d_x_scale, d_topk_weights, d_recv_q,
                    d_recv_scale, scale_col_major, d_recv_w, stream) -> int:
    return int(_lib.ep_dispatch_fp8(ctypes.byref(cfg), ctypes.byref(layout), d_x, d_x_q,
                                    d_x_scale, d_topk_weights, d_recv_q, d_recv_scale,
                                    int(scale_col_major), d_recv_w, stream))


def ep_combine_epilogue(cfg, layout, d_expert_out, d_topk_weights, d_bias0, d_bias1,
                        d_recv_w, d_y, d_combined_w, stream) -> int:
    return int(_lib.ep_combine_epilogue(ctypes.byref(cfg), ctypes.byref(layout),
                                        d_expert_out, d_topk_weights, d_bias0, d_bias1,
                                        d_recv_w, d_y, d_combined_w, stream))


def ep_dispatch_backward(cfg, layout, d_grad_recv, d_grad_recv_w, d_grad_x, d_grad_w,
                         stream) -> int:
    return int(_lib.ep_dispatch_backward(ctypes.byref(cfg), ctypes.byref(layout),
                                         d_grad_recv, d_grad_recv_w, d_grad_x, d_grad_w,
                                         stream))


def ep_combine_backward(cfg, layout, d_dy, d_topk_weights, d_expert_out,
                        d_grad_expert_out, d_grad_w, stream) -> int:
    return int(_lib.ep_combine_backward(ctypes.byref(cfg), ctypes.byref(layout), d_dy,
                                        d_topk_weights, d_expert_out, d_grad_expert_out,
                                        d_grad_w, stream))


def ep_rank_rows_capacity(cfg: EpConfig) -> int:
    return int(_lib.ep_rank_rows_capacity(ctypes.byref(cfg)))


def ep_dispatch_ranks(cfg, layout, d_x, d_topk_idx, d_topk_weights, d_rank_x,
                      d_rank_topk_idx, d_rank_topk_w, stream) -> int:
    return int(_lib.ep_dispatch_ranks(ctypes.byref(cfg), ctypes.byref(layout), d_x,
                                      d_topk_idx, d_topk_weights, d_rank_x,
                                      d_rank_topk_idx, d_rank_topk_w, stream))


def ep_expand(cfg, layout, d_topk_idx, d_rank_x, d_rank_topk_w, d_recv_x, d_recv_w,
              stream) -> int:
    return int(_lib.ep_expand(ctypes.byref(cfg), ctypes.byref(layout), d_topk_idx,
                              d_rank_x, d_rank_topk_w, d_recv_x, d_recv_w, stream))


def ep_reduce_ranks(cfg, layout, d_topk_idx, d_expert_out, d_topk_weights, d_rank_y,
                    stream) -> int:
    return int(_lib.ep_reduce_ranks(ctypes.byref(cfg), ctypes.byref(layout), d_topk_idx,
                                    d_expert_out, d_topk_weights, d_rank_y, stream))


def ep_combine_ranks(cfg, layout, d_rank_y, d_y, stream) -> int:
    return int(_lib.ep_combine_ranks(ctypes.byref(cfg), ctypes.byref(layout), d_rank_y,
                                     d_y, stream))


def ep_layout_and_dispatch(cfg, num_tokens, d_topk_idx, layout, d_x, d_topk_weights,
                           d_recv_x, d_recv_scale, d_recv_w, stream) -> int:
    return int(_lib.ep_layout_and_dispatch(ctypes.byref(cfg), int(num_tokens), d_topk_idx,
                                           ctypes.byref(layout), d_x, d_topk_weights, d_recv_x,
                                           d_recv_scale, d_recv_w, stream))


def ep_dispatch_from_host(cfg, layout, h_x, d_x, d_topk_weights, d_recv_x, d_recv_scale,
                          d_recv_w, num_chunks, stream) -> int:
    return int(_lib.ep_dispatch_from_host(ctypes.byref(cfg), ctypes.byref(layout), h_x, d_x,
                                          d_topk_weights, d_recv_x, d_recv_scale, d_recv_w,
                                          int(num_chunks), stream))


def ep_combine_to_host(cfg, layout, d_expert_out, d_topk_weights, d_y, h_y, num_chunks,
                       stream) -> int:
    return int(_lib.ep_combine_to_host(ctypes.byref(cfg), ctypes.byref(layout), d_expert_out,
                                       d_topk_weights, d_y, h_y, int(num_chunks), stream))


def ep_check_error(layout, stream) -> int:
    return int(_lib.ep_check_error(ctypes.byref(layout), stream))


def ep_selftest_fp8_quotient(d_counts, d_first, stream) -> int:
    return int(_lib.ep_selftest_fp8_quotient(d_counts, d_first, stream))


def ep_selftest_wait_timeout(timeout_ns, d_err, stream) -> int:
    return int(_lib.ep_selftest_wait_timeout(int(timeout_ns), d_err, stream))


def ep_selftest_layout_timeout(cfg, num_tokens, d_topk_idx, layout, stall_tile, timeout_ns,
                               stream) -> int:
    return int(_lib.ep_selftest_layout_timeout(ctypes.byref(cfg), num_tokens, d_topk_idx,
                                               ctypes.byref(layout), int(stall_tile),
                                               int(timeout_ns), stream))


def ep_get_layout_noalloc(cfg, num_tokens, d_topk_idx, layout, h_expert_count,
                          stream) -> int:
    """ep_get_layout with the scratch in the library's own device memory
    (layout.workspace is ignored)."""
    return int(_lib.ep_get_layout_noalloc(ctypes.byref(cfg), num_tokens, d_topk_idx,
                                          ctypes.byref(layout), h_expert_count,
                                          stream))


def ep_last_cuda_error() -> int:
    return int(_lib.ep_last_cuda_error())


def ep_status_str(status: int) -> str:
    return _lib.ep_status_str(int(status)).decode()


# ---- torch layer ------------------------------------------------------------

class EpError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = f"{what}: {ep_status_str(status)} ({status})"
        if self.status == EP_ERR_CUDA:
            self.cuda_error = ep_last_cuda_error()
            msg += f", cudaError {self.cuda_error}"
        super().__init__(msg)


def _check(status: int, what: str):
    if status != EP_OK:
        raise EpError(status, what)


@dataclasses.dataclass(frozen=True)
class Config:
    """Mirror of ep_config (see include/ep.h)."""

    max_tokens: int
    hidden: int
    num_topk: int
    num_experts: int
    num_ranks: int
    expert_alignment: int = 128
    use_fp8_dispatch: bool = False
    zero_padding: bool = False

    def c(self) -> EpConfig:
        return EpConfig(self.max_tokens, self.hidden, self.num_topk,
                        self.num_experts, self.num_ranks, self.expert_alignment,
                        int(self.use_fp8_dispatch), int(self.zero_padding))

    @property
    def capacity(self) -> int:
        cap = ep_recv_capacity(self.c())
        if cap < 0:
            raise EpError(EP_ERR_INVALID_ARG, "config")
        return cap


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Layout:
    """Device buffers of one layout handle, allocated with torch."""

    def __init__(self, cfg: Config, device="cuda", with_ranks: bool = False):
        import torch

        self.cfg = cfg
        E, R, K, T = cfg.num_experts, cfg.num_ranks, cfg.num_topk, cfg.max_tokens
        cap = cfg.capacity
        ws = ep_layout_workspace_bytes(cfg.c())
        i32 = dict(dtype=torch.int32, device=device)
        self.expert_count = torch.zeros(E, **i32)
        self.expert_start = torch.zeros(E + 1, **i32)
        self.expert_end = torch.zeros(E, **i32)
        self.rank_start = torch.zeros(R + 1, **i32)
        self.tokens_per_rank = torch.zeros(R, **i32)
        self.is_token_in_rank = torch.zeros((max(T, 1), R), dtype=torch.uint8, device=device)
        self.slot_of = torch.full((max(T, 1), K), -1, **i32)
        self.src_info = torch.full((cap, 2), -1, **i32)
        self.err = torch.zeros(4, **i32)
        self.workspace = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
        self.rank_row_start = self.rank_slot_of = self.rank_src = None
        if with_ranks:
            self.rank_row_start = torch.zeros(R + 1, **i32)
            self.rank_slot_of = torch.full((max(T, 1), R), -1, **i32)
            self.rank_src = torch.full((max(T * min(K, R), 1),), -1, **i32)
        self.c = EpLayout(
            _ptr(self.expert_count), _ptr(self.expert_start), _ptr(self.expert_end),
            _ptr(self.rank_start), _ptr(self.tokens_per_rank),
            _ptr(self.is_token_in_rank), _ptr(self.slot_of), _ptr(self.src_info),
            _ptr(self.err), _ptr(self.workspace), _ptr(self.rank_row_start),
            _ptr(self.rank_slot_of), _ptr(self.rank_src), 0, 0)

    @property
    def num_tokens(self) -> int:
        return int(self.c.num_tokens)


def get_layout(cfg: Config, topk_idx, layout: Optional[Layout] = None,
               sync: bool = False, stream=None, with_ranks: bool = False) -> Layout:
    """ep_get_layout on an int64 CUDA tensor [T, K]."""
    import numpy as np

    if layout is None:
        layout = Layout(cfg, device=topk_idx.device, with_ranks=with_ranks)
    T = int(topk_idx.shape[0])
    h = None
    if sync:
        h = np.zeros(cfg.num_experts, np.int32)
    st = ep_get_layout(cfg.c(), T, _ptr(topk_idx.contiguous()) if T else None,
                       layout.c, None if h is None else h.ctypes.data_as(ctypes.c_void_p),
                       _stream(stream))
    _check(st, "ep_get_layout")
    layout.h_expert_count = h
    return layout


def dispatch(cfg: Config, layout: Layout, x, topk_weights=None, recv_x=None,
             recv_scale=None, recv_w=None, want_weights: bool = True, stream=None):
    """ep_dispatch.  x: bf16 CUDA tensor [T, H].  Returns (recv_x, recv_scale,
    recv_w); recv_x is bf16 [cap, H] or uint8 (E4M3 bits) [cap, H]."""
    import torch

    cap, H = cfg.capacity, cfg.hidden
    dev = x.device
    if recv_x is None:
        dt = torch.uint8 if cfg.use_fp8_dispatch else torch.bfloat16
        recv_x = torch.empty((cap, H), dtype=dt, device=dev)
    if cfg.use_fp8_dispatch and recv_scale is None:
        recv_scale = torch.empty((cap, H // 128), dtype=torch.float32, device=dev)
    if want_weights and topk_weights is not None and recv_w is None:
        recv_w = torch.empty(cap, dtype=torch.float32, device=dev)
    st = ep_dispatch(cfg.c(), layout.c, _ptr(x), _ptr(topk_weights), _ptr(recv_x),
                     _ptr(recv_scale), _ptr(recv_w), _stream(stream))
    _check(st, "ep_dispatch")
    return recv_x, recv_scale, recv_w


def combine(cfg: Config, layout: Layout, expert_out, topk_weights=None, y=None,
            stream=None):
    """ep_combine.  expert_out: bf16 CUDA tensor [cap, H]; returns bf16 [T, H]."""
    import torch

    T = layout.num_tokens
    if y is None:
        y = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=expert_out.device)
    st = ep_combine(cfg.c(), layout.c, _ptr(expert_out), _ptr(topk_weights),
                    _ptr(y), _stream(stream))
    _check(st, "ep_combine")
    return y


def layout_and_dispatch(cfg: Config, topk_idx, x, topk_weights=None, layout=None,
                        recv_x=None, recv_scale=None, recv_w=None, want_weights: bool = True,
                        stream=None):
    """ep_layout_and_dispatch.  topk_idx: int64 CUDA tensor [T, K]; x: bf16 CUDA
    tensor [T, H].  Returns (layout, recv_x, recv_scale, recv_w)."""
    import torch

    cap, H = cfg.capacity, cfg.hidden
    dev = x.device
    L = layout or Layout(cfg, device=dev)
    if recv_x is None:
        dt = torch.uint8 if cfg.use_fp8_dispatch else torch.bfloat16
        recv_x = torch.empty((cap, H), dtype=dt, device=dev)
    if cfg.use_fp8_dispatch and recv_scale is None:
        recv_scale = torch.empty((cap, H // 128), dtype=torch.float32, device=dev)
    if want_weights and topk_weights is not None and recv_w is None:
        recv_w = torch.empty(cap, dtype=torch.float32, device=dev)
    st = ep_layout_and_dispatch(cfg.c(), topk_idx.shape[0], _ptr(topk_idx), L.c, _ptr(x),
                                _ptr(topk_weights), _ptr(recv_x), _ptr(recv_scale),
                                _ptr(recv_w), _stream(stream))
    _check(st, "ep_layout_and_dispatch")
    return L, recv_x, recv_scale, recv_w


def dispatch_from_host(cfg: Config, layout: Layout, h_x, d_x=None, topk_weights=None,
                       recv_x=None, recv_scale=None, recv_w=None, want_weights: bool = True,
                       num_chunks: int = 8, stream=None):
    """ep_dispatch_from_host.  h_x: bf16 CPU tensor [T, H] (pinned for overlap);
    d_x: CUDA staging tensor [T, H] (allocated when None).  num_chunks=0: the
    kernel reads h_x in place (h_x must be pinned; no staging, d_x stays
    None).  Returns (recv_x, recv_scale, recv_w, d_x)."""
    import torch

    cap, H = cfg.capacity, cfg.hidden
    dev = torch.device("cuda", torch.cuda.current_device())
    if d_x is None and num_chunks != 0:
        d_x = torch.empty(tuple(h_x.shape), dtype=torch.bfloat16, device=dev)
    if recv_x is None:
        dt = torch.uint8 if cfg.use_fp8_dispatch else torch.bfloat16
        recv_x = torch.empty((cap, H), dtype=dt, device=dev)
    if cfg.use_fp8_dispatch and recv_scale is None:
        recv_scale = torch.empty((cap, H // 128), dtype=torch.float32, device=dev)
    if want_weights and topk_weights is not None and recv_w is None:
        recv_w = torch.empty(cap, dtype=torch.float32, device=dev)
    st = ep_dispatch_from_host(cfg.c(), layout.c, _ptr(h_x), _ptr(d_x), _ptr(topk_weights),
                               _ptr(recv_x), _ptr(recv_scale), _ptr(recv_w), num_chunks,
                               _stream(stream))
    _check(st, "ep_dispatch_from_host")
    return recv_x, recv_scale, recv_w, d_x


def combine_to_host(cfg: Config, layout: Layout, expert_out, topk_weights=None, h_y=None,
                    d_y=None, num_chunks: int = 8, stream=None):
    """ep_combine_to_host.  Returns (h_y, d_y): h_y a pinned bf16 CPU tensor
    [T, H], readable once the stream has been synchronised.  num_chunks=0:
    the kernel writes h_y in place (h_y must be pinned; d_y stays None)."""
    import torch

    T, H = layout.num_tokens, cfg.hidden
    if h_y is None:
        h_y = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    if d_y is None and num_chunks != 0:
        d_y = torch.empty((T, H), dtype=torch.bfloat16, device=expert_out.device)
    st = ep_combine_to_host(cfg.c(), layout.c, _ptr(expert_out), _ptr(topk_weights), _ptr(d_y),
                            _ptr(h_y), num_chunks, _stream(stream))
    _check(st, "ep_combine_to_host")
    return h_y, d_y


def check_error(layout: Layout, stream=None) -> int:
    return ep_check_error(layout.c, _stream(stream))


def dispatch_fp8(cfg: Config, layout: Layout, x=None, x_q=None, x_scale=None,
                 topk_weights=None, scale_col_major: bool = False, recv_q=None,
                 recv_scale=None, recv_w=None, want_weights: bool = True, stream=None):
    """ep_dispatch_fp8: quantise bf16 `x`, or copy pre-quantised `x_q` (uint8
    E4M3 bits [T, H]) with `x_scale` (fp32 [T, H/128]).  Returns (recv_q,
    recv_scale, recv_w); recv_scale is [cap, H/128], or [H/128, ld] when
    scale_col_major."""
    import torch

    cap, H = cfg.capacity, cfg.hidden
    dev = (x if x is not None else x_q).device
    if recv_q is None:
        recv_q = torch.empty((cap, H), dtype=torch.uint8, device=dev)
    if recv_scale is None:
        shape = (H // 128, ep_scale_ld(cfg.c())) if scale_col_major else (cap, H // 128)
        recv_scale = torch.empty(shape, dtype=torch.float32, device=dev)
    if want_weights and topk_weights is not None and recv_w is None:
        recv_w = torch.empty(cap, dtype=torch.float32, device=dev)
    st = ep_dispatch_fp8(cfg.c(), layout.c, _ptr(x), _ptr(x_q), _ptr(x_scale),
                         _ptr(topk_weights), _ptr(recv_q), _ptr(recv_scale),
                         scale_col_major, _ptr(recv_w), _stream(stream))
    _check(st, "ep_dispatch_fp8")
    return recv_q, recv_scale, recv_w


def combine_epilogue(cfg: Config, layout: Layout, expert_out, topk_weights=None,
                     bias0=None, bias1=None, recv_w=None, want_weights: bool = False,
                     y=None, stream=None):
    """ep_combine_epilogue.  Returns (y, combined_w or None)."""
    import torch

    T = layout.num_tokens
    dev = expert_out.device
    if y is None:
        y = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=dev)
    cw = None
    if want_weights:
        cw = torch.empty((max(T, 1), cfg.num_topk), dtype=torch.float32, device=dev)
    st = ep_combine_epilogue(cfg.c(), layout.c, _ptr(expert_out), _ptr(topk_weights),
                             _ptr(bias0), _ptr(bias1), _ptr(recv_w), _ptr(y), _ptr(cw),
                             _stream(stream))
    _check(st, "ep_combine_epilogue")
    return y, (None if cw is None else cw[:T])


def dispatch_backward(cfg: Config, layout: Layout, grad_recv, grad_recv_w=None,
                      grad_x=None, stream=None):
    """ep_dispatch_backward.  Returns (grad_x bf16 [T, H], grad_w or None)."""
    import torch

    T = layout.num_tokens
    dev = grad_recv.device
    if grad_x is None:
        grad_x = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=dev)
    gw = None
    if grad_recv_w is not None:
        gw = torch.empty((max(T, 1), cfg.num_topk), dtype=torch.float32, device=dev)
    st = ep_dispatch_backward(cfg.c(), layout.c, _ptr(grad_recv), _ptr(grad_recv_w),
                              _ptr(grad_x), _ptr(gw), _stream(stream))
    _check(st, "ep_dispatch_backward")
    return grad_x, (None if gw is None else gw[:T])


def combine_backward(cfg: Config, layout: Layout, dy, topk_weights=None, expert_out=None,
                     grad_expert_out=None, want_grad_w: bool = True, stream=None):
    """ep_combine_backward.  Returns (grad_expert_out bf16 [cap, H], grad_w or
    None); grad_w needs the forward expert rows `expert_out`."""
    import torch

    T = layout.num_tokens
    dev = dy.device
    if grad_expert_out is None:
        grad_expert_out = torch.empty((cfg.capacity, cfg.hidden), dtype=torch.bfloat16,
                                      device=dev)
    gw = None
    if want_grad_w and expert_out is not None:
        gw = torch.empty((max(T, 1), cfg.num_topk), dtype=torch.float32, device=dev)
    st = ep_combine_backward(cfg.c(), layout.c, _ptr(dy), _ptr(topk_weights),
                             _ptr(expert_out), _ptr(grad_expert_out), _ptr(gw),
                             _stream(stream))
    _check(st, "ep_combine_backward")
    return grad_expert_out, (None if gw is None else gw[:T])


# ---- non-expanded (destination-major) stage ------------------------------------

def dispatch_ranks(cfg: Config, layout: Layout, x, topk_idx, topk_weights=None,
                   stream=None):
    """ep_dispatch_ranks.  Returns (rank_x bf16 [rows_cap, H], rank_topk_idx
    int32 [rows_cap, K], rank_topk_w fp32 [rows_cap, K] or None)."""
    import torch

    n = ep_rank_rows_capacity(cfg.c())
    dev = x.device
    rank_x = torch.empty((max(n, 1), cfg.hidden), dtype=torch.bfloat16, device=dev)
    ridx = torch.empty((max(n, 1), cfg.num_topk), dtype=torch.int32, device=dev)
    rw = None
    if topk_weights is not None:
        rw = torch.empty((max(n, 1), cfg.num_topk), dtype=torch.float32, device=dev)
    st = ep_dispatch_ranks(cfg.c(), layout.c, _ptr(x), _ptr(topk_idx), _ptr(topk_weights),
                           _ptr(rank_x), _ptr(ridx), _ptr(rw), _stream(stream))
    _check(st, "ep_dispatch_ranks")
    return rank_x, ridx, rw


def expand(cfg: Config, layout: Layout, topk_idx, rank_x, rank_topk_w=None,
           recv_x=None, stream=None):
    """ep_expand.  Returns (recv_x bf16 [cap, H], recv_w or None)."""
    import torch

    dev = rank_x.device
    if recv_x is None:
        recv_x = torch.empty((cfg.capacity, cfg.hidden), dtype=torch.bfloat16, device=dev)
    rw = None
    if rank_topk_w is not None:
        rw = torch.empty(cfg.capacity, dtype=torch.float32, device=dev)
    st = ep_expand(cfg.c(), layout.c, _ptr(topk_idx), _ptr(rank_x), _ptr(rank_topk_w),
                   _ptr(recv_x), _ptr(rw), _stream(stream))
    _check(st, "ep_expand")
    return recv_x, rw


def reduce_ranks(cfg: Config, layout: Layout, topk_idx, expert_out, topk_weights=None,
                 stream=None):
    """ep_reduce_ranks.  Returns rank_y bf16 [rows_cap, H]."""
    import torch

    n = ep_rank_rows_capacity(cfg.c())
    rank_y = torch.empty((max(n, 1), cfg.hidden), dtype=torch.bfloat16,
                         device=expert_out.device)
    st = ep_reduce_ranks(cfg.c(), layout.c, _ptr(topk_idx), _ptr(expert_out),
                         _ptr(topk_weights), _ptr(rank_y), _stream(stream))
    _check(st, "ep_reduce_ranks")
    return rank_y


def combine_ranks(cfg: Config, layout: Layout, rank_y, y=None, stream=None):
    """ep_combine_ranks.  Returns y bf16 [T, H]."""
    import torch

    if y is None:
        y = torch.empty((layout.num_tokens, cfg.hidden), dtype=torch.bfloat16,
                        device=rank_y.device)
    st = ep_combine_ranks(cfg.c(), layout.c, _ptr(rank_y), _ptr(y), _stream(stream))
    _check(st, "ep_combine_ranks")
    return y
